// parallel_tc.cu -- the parallel form of retention on the sm_103a tensor cores.
//
// "1. The Parallel Representation for High-Throughput Pretraining" of "RetNet
// Guide: Retentive Networks & The Impossible Triangle":
//
//   O = ((Q K^T) (.) D) V,   D[n][m] = gamma^(n-m) for n >= m, 0 otherwise,
//
// with the query factor 1/sqrt(dk) of "1. PyTorch Implementation of
// MultiScaleRetention".  Unlike softmax attention there is no running
// normaliser: every key tile adds P~_j V_j to one accumulator, which stays in
// tensor memory for the whole key loop.
//
// One CTA takes one (query tile i of 128 rows, head, value tile) and walks the
// key tiles j <= i.  Per key tile:
//   S_j  = Q_i K_j^T                    tcgen05.mma, bf16 operands from
//                                       128B-swizzled shared memory (TMA),
//                                       fp32 in tensor memory (two buffers)
//   P~_j = (S_j (.) D_ij) / sqrt(dk)    in registers, written back as bf16 in
//                                       place (the A operand of the next MMA)
//   O   += P~_j V_j                     tcgen05.mma, A from tensor memory
// The decay of element (r, c) of tile pair (i, j), Delta = i - j, is
// gamma^(Delta*128 + r - c).  On the diagonal tile it is read from a table of
// gamma^d, d < 128 (zero above the diagonal).  Off the diagonal it is the
// product of a row factor gamma^((Delta-1)*128 + 1 + r) and a column factor
// gamma^(127 - c), both at most 1, so neither factor can overflow and the
// decay is never split as gamma^n * gamma^-m.  A key tile is skipped only
// when its largest decay factor, gamma^((Delta-1)*128 + 1), is exactly 0 in
// fp32: every product it would add is then exactly 0.
//
// Roles in a CTA of 192 threads:
//   warp 0 lane 0 : TMA producer: Q_i once, then K_j and V_j into a ring
//   warp 1        : owns the TMEM allocation; lane 0 issues the MMAs in the
//                   order S_j, then O += P~_{j-1} V_{j-1}, so the tensor pipe
//                   computes S_j while the epilogue masks S_{j-1}
//   warps 2..5    : epilogue: decay and scale of S_j into P~_j; at the end
//                   the output rows, bf16, stored straight to global memory
// Every mbarrier wait gives up after 2 s, sets RET_DEV_WAIT_TIMEOUT in this
// file's device status word and unwinds (loads and MMAs in flight are waited
// for, with the same limit, before the tensor memory is released).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "retention.h"

namespace ret {

// Device status word of the parallel kernels (retention_device_status ORs it in).
__device__ unsigned int g_parallel_status = 0;

namespace {

using namespace ptx;

constexpr int kT = 128;          // rows of a query tile and of a key tile
constexpr int kPThreads = 192;
constexpr int kEpi = 128;        // epilogue threads
constexpr uint64_t kPWaitNs = 2000000000ull;

template <int DK, int DVT>
struct PCfg {
  static_assert(DK == 128 || DK == 256, "dk tile");
  static_assert(DVT == 64 || DVT == 128 || DVT == 256, "value tile");
  static constexpr int H = DK / 128;       // 128-column halves of Q and K
  static constexpr int kQ = kT * DK * 2;   // Q_i: H halves of two 64-column boxes
  static constexpr int kK = kT * DK * 2;   // K_j, same layout
  static constexpr int kV = kT * DVT * 2;  // V_j: DVT/64 boxes of 64 columns
  static constexpr int kStage = kK + kV;
  static constexpr int kTail = 2 * kT * 4 + 32 * 8 + 16;  // tables, barriers, slot, abort flag
  static constexpr int pick_ns() {
    int n = 4;
    while (n > 1 && kQ + n * kStage + kTail + 1024 > kMaxSmemPerBlock) --n;
    return n;
  }
  static constexpr int NS = pick_ns();
  static_assert(NS >= 2, "at least two stages");
  static constexpr int oK = kQ;  // stage s: K at oK + s*kStage, V right after it
  static constexpr int oPw = kQ + NS * kStage;  // pw[d] = gamma^d, d < kT
  static constexpr int oCol = oPw + kT * 4;     // colf[c] = gamma^(kT-1-c)
  static constexpr int oBar = oCol + kT * 4;
  static constexpr int oSlot = oBar + 32 * 8;
  static constexpr int oAbort = oSlot + 4;
  static constexpr int kAlloc = oAbort + 12 + 1024;
  static_assert(kAlloc <= kMaxSmemPerBlock, "shared memory");
  static_assert(kQ % 1024 == 0 && kK % 1024 == 0 && kV % 1024 == 0, "align");
  // barriers
  static constexpr int bQ = 0, bKFull = 1, bVFull = 1 + NS, bEmpty = 1 + 2 * NS, bSFull = 1 + 3 * NS,
                       bPReady = bSFull + 2, bSFree = bPReady + 2, bOFull = bSFree + 2, bFin = bOFull + 1,
                       kBars = bFin + 1;
  static_assert(kBars <= 32, "barriers");
  // tensor memory: two S buffers of kT columns, then O
  static constexpr int cS = 0, cO = 2 * kT;
  static_assert(cO + DVT <= 512, "tmem");
  static constexpr int kTmemCols = 512;
};

struct PParams {
  const float* gamma;
  __nv_bfloat16* out;  // [BH][N][dv]
  int H, N, dv, BH, n_dv_tiles, n_tiles;
  float scale;
};

__device__ __forceinline__ float pow_gamma(float g, float lg, float d) {
  if (d == 0.0f) return 1.0f;
  if (g <= 0.0f) return 0.0f;
  return exp2f(d * lg);
}

__device__ __forceinline__ void p_flag_timeout(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_parallel_status, RET_DEV_WAIT_TIMEOUT);
}

// Wait for phase `parity` of `bar`: false if this CTA aborts or the wait timed out.
__device__ __forceinline__ bool p_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kPWaitNs) {
      p_flag_timeout(abort_flag);
      return false;
    }
  }
}

// Teardown wait: ignores the abort flag, still bounded.
__device__ __forceinline__ void p_drain(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kPWaitNs) {
      p_flag_timeout(abort_flag);
      return;
    }
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int DK, int DVT>
__global__ void __launch_bounds__(kPThreads, 1)
parallel_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const PParams p) {
  using L = PCfg<DK, DVT>;
  constexpr int H = L::H, NS = L::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  float* pw = reinterpret_cast<float*>(sm + L::oPw);
  float* colf = reinterpret_cast<float*>(sm + L::oCol);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::oAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::oSlot);
  auto bar = [&](int b) { return sbase + L::oBar + 8 * b; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // heaviest query tiles first: the first BH * n_dv_tiles CTAs take the last tile
  const int units = p.BH * p.n_dv_tiles;
  const int i = p.n_tiles - 1 - (int)(blockIdx.x / (unsigned)units);
  const int u = (int)(blockIdx.x % (unsigned)units);
  const int dvt = u % p.n_dv_tiles, bh = u / p.n_dv_tiles;
  const int head = bh % p.H;
  const int dv0 = dvt * DVT;
  const float g = p.gamma[head];
  const float lg = g > 0.f ? log2f(g) : 0.f;
  // First key tile with a non-zero factor: tiles Delta >= d contribute
  // exactly zero once gamma^((d-1)*kT + 1) is zero in fp32.
  int jlo = 0;
  if (g <= 0.f) {
    jlo = i;
  } else if (g < 1.f) {
    for (int d = 1; d <= i; ++d)
      if (exp2f((float)((d - 1) * kT + 1) * lg) == 0.f) {
        jlo = i - d + 1;
        break;
      }
  }
  const int nj = i - jlo + 1;  // key tiles this CTA walks (>= 1: the diagonal)

  if (threadIdx.x == 0) {
    mbar_init(bar(L::bQ), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(L::bKFull + s), 1);
      mbar_init(bar(L::bVFull + s), 1);
      mbar_init(bar(L::bEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::bSFull + b), 1);
      mbar_init(bar(L::bPReady + b), kEpi);
      mbar_init(bar(L::bSFree + b), 1);
    }
    mbar_init(bar(L::bOFull), 1);
    mbar_init(bar(L::bFin), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  for (int d = threadIdx.x; d < kT; d += kPThreads) {
    pw[d] = pow_gamma(g, lg, (float)d);
    colf[d] = pow_gamma(g, lg, (float)(kT - 1 - d));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(L::bQ), L::kQ);
#pragma unroll
      for (int hh = 0; hh < H; ++hh)
#pragma unroll
        for (int b = 0; b < 2; ++b)
          tma_load_3d(sbase + (hh * 2 + b) * kT * 128, &tmq, hh * 128 + b * 64, i * kT, bh, bar(L::bQ));
      int issued = 0;
      for (int n = 0; n < nj; ++n) {
        const int s = n % NS, k = n / NS, j = jlo + n;
        if (k > 0 && !p_wait(bar(L::bEmpty + s), (k - 1) & 1, abort_flag)) break;
        const uint32_t sk = sbase + L::oK + s * L::kStage, sv = sk + L::kK;
        mbar_arrive_expect_tx(bar(L::bKFull + s), L::kK);
#pragma unroll
        for (int hh = 0; hh < H; ++hh)
#pragma unroll
          for (int b = 0; b < 2; ++b)
            tma_load_3d(sk + (hh * 2 + b) * kT * 128, &tmk, hh * 128 + b * 64, j * kT, bh, bar(L::bKFull + s));
        mbar_arrive_expect_tx(bar(L::bVFull + s), L::kV);
#pragma unroll
        for (int b = 0; b < DVT / 64; ++b)
          tma_load_3d(sv + b * kT * 128, &tmv, dv0 + b * 64, j * kT, bh, bar(L::bVFull + s));
        issued = n + 1;
      }
      // every issued load has landed before the CTA may exit
      p_drain(bar(L::bQ), 0, abort_flag);
      for (int n = issued - 1; n >= 0 && n >= issued - NS; --n) {
        p_drain(bar(L::bKFull + n % NS), (n / NS) & 1, abort_flag);
        p_drain(bar(L::bVFull + n % NS), (n / NS) & 1, abort_flag);
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t idP = make_idesc(kT, kT, false, false);
      constexpr uint32_t idO = make_idesc(kT, DVT, false, true);
      const uint64_t dQ = make_sdesc(sbase, 16, 1024);                   // Q, K-major A
      const uint64_t dK = make_sdesc(sbase + L::oK, 16, 1024);           // K_j, K-major B (stage 0)
      const uint64_t dV = make_sdesc(sbase + L::oK + L::kK, kT * 128, 1024);  // V_j, MN-major B (stage 0)
      constexpr uint32_t kStage16 = L::kStage >> 4;
      auto kstep = [](int hh, int kk) {  // byte offset of K-step kk of half hh in a Q or K tile
        return (uint32_t)(hh * kT * 256 + (kk >> 2) * kT * 128 + (kk & 3) * 32) >> 4;
      };
      bool ok = p_wait(bar(L::bQ), 0, abort_flag);
      auto issue_pv = [&](int m) -> bool {
        const int b = m & 1, s = m % NS;
        if (!p_wait(bar(L::bPReady + b), (m >> 1) & 1, abort_flag)) return false;
        if (!p_wait(bar(L::bVFull + s), (m / NS) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t aP = tmem + L::cS + b * kT, dO = tmem + L::cO;
        const uint64_t db = dV + (uint64_t)s * kStage16;
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk) mma_bf16_ta(dO, aP + kk * 8, db + kk * 128, idO, (m > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::bEmpty + s));   // K_m and V_m are no longer read
        mma_commit(bar(L::bSFree + b));   // nor is P~_m
        return true;
      };
      for (int n = 0; n < nj && ok; ++n) {
        const int b = n & 1, s = n % NS;
        if (n >= 2 && !p_wait(bar(L::bSFree + b), ((n - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
        if (!p_wait(bar(L::bKFull + s), (n / NS) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint64_t dk_s = dK + (uint64_t)s * kStage16;
#pragma unroll
        for (int hh = 0; hh < H; ++hh)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16(tmem + L::cS + b * kT, dQ + kstep(hh, kk), dk_s + kstep(hh, kk), idP, (hh > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(L::bSFull + b));
        if (n >= 1) ok = issue_pv(n - 1);
      }
      if (ok) ok = issue_pv(nj - 1);
      if (ok) mma_commit(bar(L::bOFull));
      // every MMA issued has completed before the tensor memory is released
      mma_commit(bar(L::bFin));
      p_drain(bar(L::bFin), 0, abort_flag);
    }
  } else {
    // ================= epilogue (warps 2..5) =================
    const int quarter = warp & 3;
    const uint32_t lane_addr = (uint32_t)(32 * quarter) << 16;
    const int r = 32 * quarter + lane;  // row of the query tile held by this thread
    auto gw = [&](uint32_t b, uint32_t parity) {
      const bool ok = p_wait(b, parity, abort_flag);
      return __all_sync(0xffffffffu, ok && !*abort_flag);
    };
    bool alive = true;
    for (int n = 0; n < nj && alive; ++n) {
      const int b = n & 1, delta = i - (jlo + n);
      if (!gw(bar(L::bSFull + b), (n >> 1) & 1)) { alive = false; break; }
      tc_fence_after();
      const uint32_t tS = tmem + lane_addr + L::cS + b * kT;
      // off the diagonal: decay = rowf * colf[c] with rowf = gamma^((delta-1)*kT + 1 + r), times the scale
      const float rowf = delta > 0 ? p.scale * pow_gamma(g, lg, (float)((delta - 1) * kT + 1 + r)) : 0.f;
#pragma unroll 1
      for (int cb = 0; cb < kT / 32; cb += 2) {
        uint32_t x[64];
        tmem_ld32p(tS + cb * 32, &x[0]);
        tmem_ld32p(tS + cb * 32 + 32, &x[32]);
        tmem_wait_ld();
        uint32_t pk[32];
        if (delta > 0) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const float2 cf = *reinterpret_cast<const float2*>(colf + cb * 32 + 2 * jj);
            pk[jj] = pack2(__uint_as_float(x[2 * jj]) * (rowf * cf.x), __uint_as_float(x[2 * jj + 1]) * (rowf * cf.y));
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int c0 = cb * 32 + 2 * jj;
            const float a = c0 <= r ? __uint_as_float(x[2 * jj]) * (p.scale * pw[r - c0]) : 0.f;
            const float bb = c0 + 1 <= r ? __uint_as_float(x[2 * jj + 1]) * (p.scale * pw[r - c0 - 1]) : 0.f;
            pk[jj] = pack2(a, bb);
          }
        }
        // P~ columns 16*cb .. 16*cb+31 lie in S columns this thread has already read
        tmem_st16(tS + cb * 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
        tmem_st16(tS + cb * 16 + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::bPReady + b));
    }
    if (alive && gw(bar(L::bOFull), 0)) {
      tc_fence_after();
      const int row = i * kT + r;
      __nv_bfloat16* orow = p.out + ((size_t)bh * p.N + row) * p.dv;
#pragma unroll 1
      for (int cb = 0; cb < DVT / 32; cb += 2) {
        uint32_t x[64];
        tmem_ld32p(tmem + lane_addr + L::cO + cb * 32, &x[0]);
        tmem_ld32p(tmem + lane_addr + L::cO + cb * 32 + 32, &x[32]);
        tmem_wait_ld();
        if (row < p.N) {
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int col = dv0 + cb * 32 + 8 * t;
            if (col < p.dv)
              *reinterpret_cast<uint4*>(orow + col) =
                  make_uint4(pack2(__uint_as_float(x[8 * t]), __uint_as_float(x[8 * t + 1])),
                             pack2(__uint_as_float(x[8 * t + 2]), __uint_as_float(x[8 * t + 3])),
                             pack2(__uint_as_float(x[8 * t + 4]), __uint_as_float(x[8 * t + 5])),
                             pack2(__uint_as_float(x[8 * t + 6]), __uint_as_float(x[8 * t + 7])));
          }
        }
      }
    }
  }

  // ---- teardown: every MMA has completed and every load landed ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int DK, int DVT>
cudaError_t launch_par(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const PParams& p,
                       cudaStream_t s) {
  using L = PCfg<DK, DVT>;
  auto kern = parallel_tc_kernel<DK, DVT>;
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  const long long grid = (long long)p.n_tiles * p.BH * p.n_dv_tiles;
  kern<<<(unsigned)grid, kPThreads, L::kAlloc, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

bool parallel_tc_supported(int dk, int dv) {
  return dk % 16 == 0 && dv % 16 == 0 && dk >= 16 && dv >= 16 && dk <= 256 && dv <= 1024;
}

cudaError_t launch_parallel_tc(const void* q, const void* k, const void* v, const float* gamma, void* out, int B,
                               int H, int N, int dk, int dv, cudaStream_t s) {
  const int BH = B * H;
  const int DK = dk <= 128 ? 128 : 256;
  const int DVT = DK == 256 ? 64 : (dv <= 64 ? 64 : (dv <= 128 ? 128 : 256));
  PParams p;
  p.gamma = gamma;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.H = H;
  p.N = N;
  p.dv = dv;
  p.BH = BH;
  p.n_dv_tiles = (dv + DVT - 1) / DVT;
  p.n_tiles = (N + kT - 1) / kT;
  p.scale = (float)(1.0 / std::sqrt((double)dk));
  if ((long long)p.n_tiles * BH * p.n_dv_tiles > INT32_MAX) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, dk, N, BH, kT) || !make_map(&mk, k, dk, N, BH, kT) || !make_map(&mv, v, dv, N, BH, kT))
    return cudaErrorInvalidValue;
  if (DK == 128) {
    if (DVT == 64) return launch_par<128, 64>(mq, mk, mv, p, s);
    if (DVT == 128) return launch_par<128, 128>(mq, mk, mv, p, s);
    return launch_par<128, 256>(mq, mk, mv, p, s);
  }
  return launch_par<256, 64>(mq, mk, mv, p, s);
}

cudaError_t read_parallel_status(unsigned int* flags, int clear) {
  cudaError_t e = cudaMemcpyFromSymbol(flags, g_parallel_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_parallel_status, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace ret
