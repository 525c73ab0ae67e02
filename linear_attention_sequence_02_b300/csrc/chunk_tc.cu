// chunk_tc.cu -- chunkwise retention forward on the sm_103a tensor cores.
//
// Per head (b, h) and 64- or 128-wide slab of value columns, for each chunk of
// C tokens (section "3. The Chunkwise Recurrent Representation ..." of "RetNet
// Guide: Retentive Networks & The Impossible Triangle"; the in-chunk decay of
// the state update is the reading that makes the chunkwise form equal the
// recurrent one):
//
//   P   = Q_i K_i^T                          (tcgen05, fp32 in TMEM)
//   P~  = (P (.) D_C) / sqrt(dk) -> bf16     (registers; D_C[r][c] = gamma^(r-c), r >= c)
//   W   = diag(gamma^(L-1-j)) V_i -> bf16    (shared memory)
//   O1  = Q_i S_{i-1}                        (tcgen05; S_{i-1} copied to bf16)
//   O2  = P~ V_i                             (tcgen05)
//   out = O2 + diag(gamma^(j+1)) O1 / sqrt(dk)   (registers -> bf16 -> TMA store)
//   S_i = gamma^L S_{i-1} + K_i^T W          (fp32 state kept in TMEM across chunks)
//
// Roles inside a CTA of 192 threads:
//   warp 0 lane 0 : TMA producer (Q, K, V boxes into an NS-deep stage ring)
//   warp 1        : owns the TMEM allocation; lane 0 issues every tcgen05.mma
//   warps 2..5    : epilogue; warp w reads TMEM lanes 32*(w%4) .. +31
// Every mbarrier wait gives up after kWaitLimitNs, sets RET_DEV_WAIT_TIMEOUT in
// the device status word and unwinds: in-flight TMA loads and MMAs are waited
// for (again with a limit), bulk stores drained and TMEM released.
//
// Long sequences are cut into `segments` runs of chunks so that enough CTAs
// exist to fill the GPU.  A state-only pre-pass (the same kernel without Q, P
// or outputs) writes each segment's local end state to a float32 workspace;
// the main pass starts segment s from sum_{t<s} gamma^((s-1-t) Lseg) state_t,
// the exclusive scan of (gamma^Lseg, state_t) pairs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "retention.h"

namespace ret {

// Device status word read by retention_device_status.
__device__ unsigned int g_device_status = 0;

namespace {

using namespace ptx;

constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kEpiBarrier = 1;                 // named barrier id of the epilogue warps
constexpr uint64_t kWaitLimitNs = 2000000000ull;    // 2 s per wait

// Rows of an M=64 accumulator occupy the first 16 lanes of each 32-lane TMEM
// sub-partition: row 16*q + l lives in lane 32*q + l, l < 16.
__device__ __forceinline__ int acc_row(int M, int quarter, int lane) {
  if (M == 128) return 32 * quarter + lane;
  return lane < 16 ? 16 * quarter + lane : -1;
}

template <int C, int DK, int DVT, int NS, bool SO>
struct Cfg {
  static_assert(C == 64 || C == 128, "chunk");
  static_assert(DK == 128 || DK == 256, "dk");
  static_assert(DVT == 64 || DVT == 128, "value tile");
  static constexpr int kQ = SO ? 0 : C * DK * 2;
  static constexpr int kK = C * DK * 2;
  static constexpr int kV = C * DVT * 2;
  static constexpr int kStage = kQ + kK + kV;
  static constexpr int kW = C * DVT * 2;
  static constexpr int kP = SO ? 0 : C * C * 2;
  static constexpr int kSb = SO ? 0 : DK * DVT * 2;
  static constexpr bool kOsAlias = !SO && DVT <= C;  // output staging reuses the P~ buffer
  static constexpr int kOs = (SO || kOsAlias) ? 0 : C * DVT * 2;
  static constexpr int oW = NS * kStage;
  static constexpr int oP = oW + kW;
  static constexpr int oSb = oP + kP;
  static constexpr int oOs = kOsAlias ? oP : oSb + kSb;
  static constexpr int oPw = oSb + kSb + kOs;
  static constexpr int kPw = ((C + 1) * 4 + 15) / 16 * 16;
  static constexpr int oBar = oPw + kPw;
  // barriers: FULL[NS], EMPTY[NS], P_FULL, P_FREE, SB_READY, PW_READY, O_FULL, O_FREE, S_FULL, FIN
  static constexpr int kBars = 2 * NS + 8;
  static constexpr int oSlot = oBar + kBars * 8;
  static constexpr int oAbort = oSlot + 4;
  static constexpr int kBytes = oAbort + 4;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 bytes
  static_assert(kAlloc <= kMaxSmemPerBlock, "shared memory");
  static_assert(kStage % 1024 == 0 && kW % 1024 == 0 && kP % 1024 == 0 && kSb % 1024 == 0, "align");
  // TMEM columns
  static constexpr int kSCols = (DK / 128) * DVT;
  static constexpr int cS = 0, cP = kSCols, cO1 = kSCols + C, cO2 = kSCols + C + DVT;
  static constexpr int kColsUsed = SO ? kSCols : kSCols + C + 2 * DVT;
  static constexpr int kTmemCols = kColsUsed <= 32 ? 32 : kColsUsed <= 64 ? 64 : kColsUsed <= 128 ? 128
                                   : kColsUsed <= 256 ? 256 : 512;
  static_assert(kColsUsed <= 512, "tmem");
  // barrier indices
  static constexpr int bFull = 0, bEmpty = NS, bPFull = 2 * NS, bPFree = 2 * NS + 1,
                       bSbReady = 2 * NS + 2, bPwReady = 2 * NS + 3, bOFull = 2 * NS + 4,
                       bOFree = 2 * NS + 5, bSFull = 2 * NS + 6, bFin = 2 * NS + 7;
};

struct TcParams {
  const float* gamma;
  float* state_out;  // main pass: final state (may be null); pre-pass: unused
  float* ws;         // segment states [B*H][segments-1][DK][dv]
  int H, N, dv, n_dv_tiles, segments, seg_chunks, n_chunks;
  float scale;       // 1/sqrt(dk)
};

__device__ __forceinline__ float gamma_pow(float g, float lg, float d) {
  if (d == 0.0f) return 1.0f;
  if (g <= 0.0f) return 0.0f;
  return exp2f(d * lg);
}

__device__ __forceinline__ void flag_timeout(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_device_status, RET_DEV_WAIT_TIMEOUT);
}

// Wait for phase `parity` of `bar`; false if this CTA is aborting or the wait timed out.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      flag_timeout(abort_flag);
      return false;
    }
  }
}

// Teardown wait: ignores the abort flag, still bounded.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      flag_timeout(abort_flag);
      return;
    }
  }
}

// Epilogue-wide wait: every epilogue thread waits, then all agree (one
// barrier with an OR) on whether to go on, so the warps never diverge.
__device__ __forceinline__ bool epi_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const bool ok = wait_bar(bar, parity, abort_flag);
  return !named_bar_or(kEpiBarrier, kEpiThreads, !ok || *abort_flag);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Store 32 fp32 values (columns col0..col0+31, col0 % 32 == 0) of row `row` as
// bf16 into a 128-byte-swizzled tile made of 64-column blocks of `rows_per_block` rows.
__device__ __forceinline__ void store_row32_swz(uint8_t* tile, int rows_per_block, int row, int col0,
                                                const float (&x)[32]) {
  uint8_t* blk = tile + (col0 / 64) * rows_per_block * 128;
  const int c16 = (col0 % 64) / 8;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint4 v;
    v.x = pack_bf16(x[8 * j + 0], x[8 * j + 1]);
    v.y = pack_bf16(x[8 * j + 2], x[8 * j + 3]);
    v.z = pack_bf16(x[8 * j + 4], x[8 * j + 5]);
    v.w = pack_bf16(x[8 * j + 6], x[8 * j + 7]);
    *reinterpret_cast<uint4*>(blk + swz128(row, c16 + j)) = v;
  }
}

template <int C, int DK, int DVT, int NS, bool SO>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                const TcParams p) {
  using L = Cfg<C, DK, DVT, NS, SO>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  float* pw = reinterpret_cast<float*>(sm + L::oPw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::oAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::oSlot);
  auto bar = [&](int i) { return sbase + L::oBar + 8 * i; };
  auto stage_q = [&](int s) { return sbase + s * L::kStage; };
  auto stage_k = [&](int s) { return sbase + s * L::kStage + L::kQ; };
  auto stage_v = [&](int s) { return sbase + s * L::kStage + L::kQ + L::kK; };

  // ---- work item ----
  const int segs_in_grid = SO ? p.segments - 1 : p.segments;
  int idx = blockIdx.x;
  const int dvt = idx % p.n_dv_tiles;
  idx /= p.n_dv_tiles;
  const int seg = idx % segs_in_grid;
  const int bh = idx / segs_in_grid;
  const int h = bh % p.H;
  const int c_begin = seg * p.seg_chunks;
  const int c_end = min(c_begin + p.seg_chunks, p.n_chunks);
  const int nck = c_end - c_begin;
  const int dv0 = dvt * DVT;
  const float g = p.gamma[h];
  const float lg = g > 0.f ? log2f(g) : 0.f;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- set-up ----
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar(L::bFull + i), 1);
      mbar_init(bar(L::bEmpty + i), 1);
    }
    mbar_init(bar(L::bPFull), 1);
    mbar_init(bar(L::bPFree), kEpiThreads);
    mbar_init(bar(L::bSbReady), kEpiThreads);
    mbar_init(bar(L::bPwReady), kEpiThreads);
    mbar_init(bar(L::bOFull), 1);
    mbar_init(bar(L::bOFree), kEpiThreads);
    mbar_init(bar(L::bSFull), 1);
    mbar_init(bar(L::bFin), 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (!SO) prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
    if (!SO) prefetch_tensormap(&tmo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  for (int d = threadIdx.x; d <= C; d += kThreads) pw[d] = gamma_pow(g, lg, (float)d);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      int issued = 0;
      for (int li = 0; li < nck; ++li) {
        const int s = li % NS, n = li / NS;
        if (li >= NS && !wait_bar(bar(L::bEmpty + s), (n - 1) & 1, abort_flag)) break;
        const int row = (c_begin + li) * C;
        mbar_arrive_expect_tx(bar(L::bFull + s), L::kStage);
        if (!SO) {
#pragma unroll
          for (int b = 0; b < DK / 64; ++b)
            tma_load_3d(stage_q(s) + b * C * 128, &tmq, b * 64, row, bh, bar(L::bFull + s));
        }
#pragma unroll
        for (int b = 0; b < DK / 64; ++b)
          tma_load_3d(stage_k(s) + b * C * 128, &tmk, b * 64, row, bh, bar(L::bFull + s));
#pragma unroll
        for (int b = 0; b < DVT / 64; ++b)
          tma_load_3d(stage_v(s) + b * C * 128, &tmv, dv0 + b * 64, row, bh, bar(L::bFull + s));
        issued = li + 1;
      }
      // every issued load has landed before the CTA may exit
      for (int li = issued - 1; li >= 0 && li >= issued - NS; --li)
        drain_bar(bar(L::bFull + li % NS), (li / NS) & 1, abort_flag);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t idP = make_idesc(C, C, false, false);
      constexpr uint32_t idO = make_idesc(C, DVT, false, true);
      constexpr uint32_t idS = make_idesc(128, DVT, true, true);
      const uint32_t sW = sbase + L::oW, sP = sbase + L::oP, sSb = sbase + L::oSb;
      for (int li = 0; li < nck; ++li) {
        const int s = li % NS, n = li / NS;
        if (!wait_bar(bar(L::bFull + s), n & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t sQ = stage_q(s), sK = stage_k(s), sV = stage_v(s);
        if (!SO) {
          if (li > 0 && !wait_bar(bar(L::bPFree), (li - 1) & 1, abort_flag)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t off = (kk / 4) * C * 128 + (kk % 4) * 32;
            mma_bf16(tmem + L::cP, make_sdesc(sQ + off, 16, 1024), make_sdesc(sK + off, 16, 1024), idP,
                     kk > 0);
          }
          mma_commit(bar(L::bPFull));
          if (!wait_bar(bar(L::bSbReady), li & 1, abort_flag)) break;
          if (li > 0 && !wait_bar(bar(L::bOFree), (li - 1) & 1, abort_flag)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < DK / 16; ++kk) {
            const uint32_t aoff = (kk / 4) * C * 128 + (kk % 4) * 32;
            mma_bf16(tmem + L::cO1, make_sdesc(sQ + aoff, 16, 1024),
                     make_sdesc(sSb + kk * 2048, DK * 128, 1024), idO, kk > 0);
          }
          if (!wait_bar(bar(L::bPwReady), li & 1, abort_flag)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C / 16; ++kk) {
            const uint32_t aoff = (kk / 4) * C * 128 + (kk % 4) * 32;
            mma_bf16(tmem + L::cO2, make_sdesc(sP + aoff, 16, 1024),
                     make_sdesc(sV + kk * 2048, C * 128, 1024), idO, kk > 0);
          }
          mma_commit(bar(L::bOFull));
        } else {
          if (!wait_bar(bar(L::bSbReady), li & 1, abort_flag)) break;
          tc_fence_after();
        }
#pragma unroll
        for (int half = 0; half < DK / 128; ++half) {
#pragma unroll
          for (int kk = 0; kk < C / 16; ++kk) {
            mma_bf16(tmem + L::cS + half * DVT,
                     make_sdesc(sK + half * 2 * C * 128 + kk * 2048, C * 128, 1024),
                     make_sdesc(sW + kk * 2048, C * 128, 1024), idS, 1u);
          }
        }
        mma_commit(bar(L::bSFull));
        mma_commit(bar(L::bEmpty + s));
      }
      // every issued MMA has completed before TMEM is released
      mma_commit(bar(L::bFin));
      drain_bar(bar(L::bFin), 0, abort_flag);
    }
  } else {
    // ================= epilogue (warps 2..5) =================
    const int et = threadIdx.x - 64;
    const int quarter = warp & 3;
    const uint32_t lane_addr = (uint32_t)(32 * quarter) << 16;
    const int srow = 32 * quarter + lane;  // state row (and row of M=128 accumulators)
    const int arow = acc_row(C, quarter, lane);  // row of the C-row accumulators (P, O1, O2)
    const uint32_t tS = tmem + lane_addr + L::cS;
    uint8_t* sW = sm + L::oW;

    // initial state: zero, or (main pass, segment > 0) the decayed sum of the
    // preceding segments' local states
    {
      const float* ws_head = p.ws + (size_t)bh * (p.segments - 1) * DK * p.dv;
      const float seg_len = (float)p.seg_chunks * (float)C;
#pragma unroll 1
      for (int half = 0; half < DK / 128; ++half) {
        const int row = half * 128 + srow;
#pragma unroll 1
        for (int cb = 0; cb < DVT / 32; ++cb) {
          float acc[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[j] = 0.f;
          if (!SO) {
            for (int t = 0; t < seg; ++t) {
              const float f = gamma_pow(g, lg, (float)(seg - 1 - t) * seg_len);
              const float4* src = reinterpret_cast<const float4*>(
                  ws_head + ((size_t)t * DK + row) * p.dv + dv0 + cb * 32);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 x = src[j];
                acc[4 * j + 0] = fmaf(f, x.x, acc[4 * j + 0]);
                acc[4 * j + 1] = fmaf(f, x.y, acc[4 * j + 1]);
                acc[4 * j + 2] = fmaf(f, x.z, acc[4 * j + 2]);
                acc[4 * j + 3] = fmaf(f, x.w, acc[4 * j + 3]);
              }
            }
          }
          uint32_t r[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(acc[j]);
          tmem_st32(tS + half * DVT + cb * 32, r);
        }
      }
      tmem_wait_st();
    }

    bool alive = true;
    for (int li = 0; li < nck && alive; ++li) {
      const int s = li % NS, n = li / NS;
      const int row0 = (c_begin + li) * C;
      const int len = min(C, p.N - row0);
      const float gL = pw[len];

      // ---- S round trip: bf16 copy of S_{i-1} for Q S, then S <- gamma^L S ----
      if (li > 0) {
        if (!epi_wait(bar(L::bSFull), (li - 1) & 1, abort_flag)) { alive = false; break; }
        tc_fence_after();
      }
#pragma unroll 1
      for (int half = 0; half < DK / 128; ++half) {
#pragma unroll 1
        for (int cb = 0; cb < DVT / 32; ++cb) {
          uint32_t r[32];
          tmem_ld32(tS + half * DVT + cb * 32, r);
          tmem_wait_ld();
          float x[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(r[j]);
          if (!SO) store_row32_swz(sm + L::oSb, DK, half * 128 + srow, cb * 32, x);
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(x[j] * gL);
          tmem_st32(tS + half * DVT + cb * 32, r);
        }
      }
      tmem_wait_st();
      if (!SO) {
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(L::bSbReady));
      }

      // ---- W = diag(gamma^(L-1-j)) V ----
      if (!epi_wait(bar(L::bFull + s), n & 1, abort_flag)) { alive = false; break; }
      {
        const uint8_t* sV = sm + (stage_v(s) - sbase);
#pragma unroll 2
        for (int q16 = et; q16 < L::kV / 16; q16 += kEpiThreads) {
          const int off = q16 * 16;
          const int row = (off % (C * 128)) / 128;
          const float f = row < len ? pw[len - 1 - row] : 0.f;
          uint4 v = *reinterpret_cast<const uint4*>(sV + off);
          uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float2 t = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[j]));
            w[j] = pack_bf16(t.x * f, t.y * f);
          }
          *reinterpret_cast<uint4*>(sW + off) = v;
        }
      }
      fence_proxy_async_smem();
      if (SO) {
        tc_fence_before();
        mbar_arrive(bar(L::bSbReady));
        continue;
      }

      // ---- P~ = (Q K^T (.) D) / sqrt(dk) -> bf16 ----
      if (L::kOsAlias) {
        if (et == 0) bulk_wait_group_read0();  // previous output store has read the shared buffer
        named_bar_sync(kEpiBarrier, kEpiThreads);
      }
      if (!epi_wait(bar(L::bPFull), li & 1, abort_flag)) { alive = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int cb = 0; cb < C / 32; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_addr + L::cP + cb * 32, r);
        tmem_wait_ld();
        if (arow >= 0) {
          float x[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int c = cb * 32 + j;
            x[j] = (c <= arow) ? pw[arow - c] * p.scale * __uint_as_float(r[j]) : 0.f;
          }
          store_row32_swz(sm + L::oP, C, arow, cb * 32, x);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(L::bPFree));
      fence_proxy_async_smem();
      mbar_arrive(bar(L::bPwReady));

      // ---- out = O2 + diag(gamma^(j+1)) O1 / sqrt(dk) ----
      if (!epi_wait(bar(L::bOFull), li & 1, abort_flag)) { alive = false; break; }
      tc_fence_after();
      if (!L::kOsAlias) {
        if (et == 0) bulk_wait_group_read0();
        named_bar_sync(kEpiBarrier, kEpiThreads);
      }
      const float zs = arow >= 0 ? pw[arow + 1] * p.scale : 0.f;
#pragma unroll 1
      for (int cb = 0; cb < DVT / 32; ++cb) {
        uint32_t a[32], b[32];
        tmem_ld32(tmem + lane_addr + L::cO1 + cb * 32, a);
        tmem_ld32(tmem + lane_addr + L::cO2 + cb * 32, b);
        tmem_wait_ld();
        if (arow >= 0) {
          float x[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = fmaf(zs, __uint_as_float(a[j]), __uint_as_float(b[j]));
          store_row32_swz(sm + L::oOs, C, arow, cb * 32, x);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(L::bOFree));
      fence_proxy_async_smem();
      named_bar_sync(kEpiBarrier, kEpiThreads);
      if (et == 0) {
#pragma unroll
        for (int b = 0; b < DVT / 64; ++b)
          tma_store_3d(&tmo, sbase + L::oOs + b * C * 128, dv0 + b * 64, row0, bh);
        bulk_commit_group();
      }
    }

    // ---- final state of this CTA's run of chunks ----
    if (alive && nck > 0) {
      if (epi_wait(bar(L::bSFull), (nck - 1) & 1, abort_flag)) {
        tc_fence_after();
        float* dst = nullptr;
        if (SO) dst = p.ws + ((size_t)bh * (p.segments - 1) + seg) * DK * p.dv;
        else if (seg == p.segments - 1 && p.state_out) dst = p.state_out + (size_t)bh * DK * p.dv;
#pragma unroll 1
        for (int half = 0; half < DK / 128; ++half) {
#pragma unroll 1
          for (int cb = 0; cb < DVT / 32; ++cb) {
            uint32_t r[32];
            tmem_ld32(tS + half * DVT + cb * 32, r);
            tmem_wait_ld();
            if (dst) {
              float4* o = reinterpret_cast<float4*>(dst + (size_t)(half * 128 + srow) * p.dv + dv0 + cb * 32);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                o[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                   __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            }
          }
        }
      }
    }
    if (!SO && et == 0) bulk_wait_group0();
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// [BH][N][d] bf16 tensor viewed in 3-D with 64-column x `rows`-row boxes, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int d, int N, int BH, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * (cuuint64_t)N};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int C, int DK, int DVT, int NS, bool SO>
cudaError_t launch_one(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const CUtensorMap& mo, const TcParams& p, int grid, cudaStream_t s) {
  using L = Cfg<C, DK, DVT, NS, SO>;
  auto kern = chunk_tc_kernel<C, DK, DVT, NS, SO>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, L::kAlloc, s>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

template <int C, int DK, int DVT, int NS>
cudaError_t launch_pair(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const CUtensorMap& mo, const TcParams& p, int BH, cudaStream_t s) {
  if (p.segments > 1) {
    constexpr int NS_SO = NS + 1;  // the pre-pass holds no Q, P or output buffers
    cudaError_t e = launch_one<C, DK, DVT, NS_SO, true>(mq, mk, mv, mo, p,
                                                        BH * (p.segments - 1) * p.n_dv_tiles, s);
    if (e != cudaSuccess) return e;
  }
  return launch_one<C, DK, DVT, NS, false>(mq, mk, mv, mo, p, BH * p.segments * p.n_dv_tiles, s);
}

// The (chunk, dk, value-tile, stages) variants compiled into the library.
int pick_dvt(int chunk, int dk, int dv) {
  if (dk == 128 && chunk == 64 && dv % 128 == 0) return 128;
  return 64;
}

}  // namespace

bool chunk_tc_plan(int B, int H, int N, int dk, int dv, int chunk, int num_sms, ChunkPlan* plan) {
  if (!(chunk == 64 || chunk == 128)) return false;
  if (!(dk == 128 || dk == 256)) return false;
  if (dv <= 0 || dv % 64 != 0 || dv > 1024) return false;
  if (N < 0) return false;
  const int dvt = pick_dvt(chunk, dk, dv);
  plan->dvt = dvt;
  plan->n_dv_tiles = dv / dvt;
  plan->n_chunks = (N + chunk - 1) / chunk;
  const long long units = (long long)B * H * plan->n_dv_tiles;
  if (units > (1LL << 30)) return false;
  // Enough segments that every SM gets a CTA, each segment at least 4 chunks.
  int segs = 1;
  if (num_sms > 0 && units < num_sms) segs = (int)(num_sms / units);
  segs = std::max(1, std::min(segs, plan->n_chunks / 4));
  int seg_chunks = plan->n_chunks > 0 ? (plan->n_chunks + segs - 1) / segs : 1;
  if (plan->n_chunks > 0) segs = (plan->n_chunks + seg_chunks - 1) / seg_chunks;  // no empty segment
  plan->segments = std::max(1, segs);
  plan->seg_chunks = std::max(1, seg_chunks);
  plan->workspace_bytes =
      plan->segments > 1 ? sizeof(float) * (size_t)B * H * (plan->segments - 1) * dk * dv : 0;
  plan->launches = plan->segments > 1 ? 2 : 1;
  if ((long long)units * plan->segments > INT32_MAX) return false;
  return true;
}

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* gamma, void* out,
                            float* state_out, int B, int H, int N, int dk, int dv, int chunk,
                            const ChunkPlan& plan, float* workspace, cudaStream_t s) {
  const int BH = B * H;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, q, dk, N, BH, chunk) || !make_map(&mk, k, dk, N, BH, chunk) ||
      !make_map(&mv, v, dv, N, BH, chunk) || !make_map(&mo, out, dv, N, BH, chunk))
    return cudaErrorInvalidValue;
  TcParams p;
  p.gamma = gamma;
  p.state_out = state_out;
  p.ws = workspace;
  p.H = H;
  p.N = N;
  p.dv = dv;
  p.n_dv_tiles = plan.n_dv_tiles;
  p.segments = plan.segments;
  p.seg_chunks = plan.seg_chunks;
  p.n_chunks = plan.n_chunks;
  p.scale = (float)(1.0 / std::sqrt((double)dk));
  if (chunk == 64 && dk == 128 && plan.dvt == 128) return launch_pair<64, 128, 128, 2>(mq, mk, mv, mo, p, BH, s);
  if (chunk == 64 && dk == 128) return launch_pair<64, 128, 64, 2>(mq, mk, mv, mo, p, BH, s);
  if (chunk == 128 && dk == 128) return launch_pair<128, 128, 64, 2>(mq, mk, mv, mo, p, BH, s);
  if (chunk == 64 && dk == 256) return launch_pair<64, 256, 64, 2>(mq, mk, mv, mo, p, BH, s);
  if (chunk == 128 && dk == 256) return launch_pair<128, 256, 64, 1>(mq, mk, mv, mo, p, BH, s);
  return cudaErrorNotSupported;
}

cudaError_t read_device_status(unsigned int* flags, int clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(flags, g_device_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace ret
