// chunk_tc.cu -- chunkwise retention forward on the sm_103a tensor cores.
//
// One CTA handles one (head b*H+h, 64- or 128-wide slab of value columns,
// run of consecutive chunks).  For chunk i (tokens t, m = 0..L-1 inside the
// chunk, L = C except for a ragged last chunk) section "3. The Chunkwise
// Recurrent Representation ..." of "RetNet Guide: Retentive Networks & The
// Impossible Triangle" gives, with the in-chunk decay of the state update made
// explicit (the reading under which the chunkwise form equals the recurrent
// one):
//
//   out_t = scale [ sum_{m<=t} gamma^(t-m) (q_t . k_m) v_m + gamma^(t+1) q_t S_{i-1} ]
//   S_i   = gamma^L S_{i-1} + sum_m gamma^(L-1-m) k_m^T v_m          (scale = 1/sqrt(dk))
//
// Rescaled form (heads with gamma^C >= 2^-14, which includes every head of the
// schedule gamma_h = 1 - 2^(-5-h)).  The tensor memory holds S^ = c S with a
// running factor c in [1, 2).  Per chunk, n = floor(log2(c / gamma^L)) and
// c' = 2^-n c / gamma^L, and with w_m = c' gamma^(L-1-m) and W = diag(w) V:
//
//   S^_i = 2^-n S^_{i-1} + K^T W                  one MMA chain; 2^-n is the MMA's
//                                                 accumulator scale operand
//   O'   = tril(Q K^T) W + Q (2^-n S^_{i-1})      one accumulator, causal mask only
//   out_t = O'_t * scale / (c' gamma^(L-1-t))
//
// (substituting w and c' gives back the two lines above exactly).  Every
// factor lies in [gamma^(C-1), 2], so nothing overflows, and no pass over the
// state in tensor memory sits on the chunk-to-chunk chain.
//
// Direct form (any other gamma in [0, 1]): the state is decayed explicitly in
// tensor memory each chunk, P~ = (Q K^T (.) D) scale with D[t][m] = gamma^(t-m),
// and, in place in shared memory after the Q K^T product has read them,
// K <- diag(gamma^(L-1-m)) K and Q <- diag(scale gamma^(t+1)) Q, so that
//   S_i = gamma^L S_{i-1} + K^T V,   out = P~ V + Q S_{i-1}.
//
// Roles in a CTA of 352 threads:
//   warp 0 lane 0 : TMA producer: V tiles and 128-column halves of Q and K into
//                   two shared-memory rings
//   warp 1        : owns the TMEM allocation; lane 0 issues Q K^T and the
//                   state update (every MMA of the state-only pre-pass)
//   warp 10 lane 0: issues Q S and P~ W, the products accumulated into O
//   warps 2..5    : state group: W = diag(w) V in place, the bf16 snapshot of
//                   the state for the Q S product, the final state; with the
//                   output group, the initial state of a later segment
//   warps 6..9    : output group: causal mask of P = Q K^T into bf16 in place in
//                   tensor memory (the A operand of P~ W); output rows scaled
//                   (with NORM, normalised per head first), staged in shared
//                   memory (its own buffer, or the chunk's V slot when there
//                   is no room) and written by a TMA store
// Warp w (w >= 2) reads TMEM lanes 32*(w%4) .. +31.
//
// Long sequences are cut into segments so that enough CTAs fill the GPU.  A
// unit is one (head, value tile); when there are more units than SMs, only
// the units of the last, partial wave are cut (so that wave holds as many
// shorter CTAs as there are SMs), and the others run whole.  A
// state-only pre-pass (this kernel with SO = true: K and V only) writes each
// segment's local end state, sum_m gamma^(Lseg-1-m) k_m^T v_m, to a float32
// workspace.  It walks the segment from its last chunk back to its first with
// each chunk's decay in its W, so one accumulating MMA chain serves any gamma
// (no rescaled state, no direct form).  The main pass starts
// segment s from gamma^(s Lseg) state_in (the caller's starting state, if any)
// plus sum_{t<s} gamma^((s-1-t) Lseg) state_t.  The main pass is launched with
// programmatic stream serialisation: its CTAs start while the pre-pass runs
// and only the two epilogue groups of a later segment wait
// (griddepcontrol.wait) before they read the workspace.
//
// Every mbarrier wait gives up after kWaitLimitNs, sets RET_DEV_WAIT_TIMEOUT in
// the device status word and unwinds: in-flight TMA loads and MMAs are waited
// for (again with a limit), bulk stores drained and TMEM released.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "angle.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "retention.h"

namespace ret {

// Device status word read by retention_device_status.
__device__ unsigned int g_device_status = 0;

namespace {

using namespace ptx;

constexpr int kThreads = 352;
constexpr int kIssuerWarpB = 10;                  // warp of the second MMA issuer
constexpr int kGroup = 128;                         // threads of one epilogue group
constexpr uint32_t kBarO = 2;                       // named barrier of the output group
constexpr uint32_t kBarInit = 3;                    // state and output groups after the initial state
constexpr uint64_t kWaitLimitNs = 2000000000ull;    // 2 s per wait
constexpr float kMinChunkDecayLog2 = -14.0f;        // rescaled form: gamma^C >= 2^-14

// Rows of an M=64 accumulator occupy the first 16 lanes of each 32-lane TMEM
// sub-partition: row 16*q + l lives in lane 32*q + l, l < 16.
__device__ __forceinline__ int acc_row(int M, int quarter, int lane) {
  if (M == 128) return 32 * quarter + lane;
  return lane < 16 ? 16 * quarter + lane : -1;
}

template <int C, int DK, int DVT, bool SO>
struct Cfg {
  static_assert(C == 64 || C == 128, "chunk");
  static_assert(DK == 128 || DK == 256 || DK == 512, "dk");
  // 512-wide queries and keys: four 128-column halves of the state (256 TMEM
  // columns at 64-wide value tiles) and 64-token tiles, so the Q/K ring holds
  // more than one chunk
  static_assert(DK < 512 || (C == 64 && DVT == 64), "512-wide keys: 64-token tiles, 64-wide value tiles");
  static_assert(DVT == 64 || DVT == 128, "value tile");
  static constexpr int kC = C, kDVT = DVT;
  static constexpr int H = DK / 128;                  // 128-row halves of the state
  // shared memory
  static constexpr int kQ = SO ? 0 : C * 256;         // one 128-column half of Q_i: two 64-column boxes
  static constexpr int kK = C * 256;                  // the same half of K_i
  static constexpr int kQK = kQ + kK;
  static constexpr int kV = C * DVT * 2;              // V_i slab (also W_i, then the output staging)
  static constexpr int kSb = SO ? 0 : 128 * DVT * 2;  // bf16 snapshot of one state half
  static constexpr int kPw = ((C + 1) * 4 + 15) / 16 * 16;
  static constexpr int kBarBytes = 80 * 8;
  static constexpr int kStg = SO ? 0 : C * DVT * 2;   // output tile staging for the TMA store
  static constexpr int bytes(int nqk, int nv, int nsb, int nstg) {
    return nqk * kQK + nv * kV + nsb * kSb + nstg * kStg + kPw + kBarBytes + 16 + 1024;  // + slack to align
  }
  static constexpr int kMinQK = 3 > 2 * H ? 3 : 2 * H;
  // Preferred layout: its own output staging buffer and two snapshot buffers,
  // so that neither V slots nor snapshots wait for output stores; else its own
  // staging buffer and one snapshot buffer; else (no room) the output tile is
  // staged in the chunk's V slot.
  static constexpr bool kSepStage = !SO && bytes(kMinQK, 3, 1, 1) <= kMaxSmemPerBlock;
  static constexpr int NSB = !SO && kSepStage && bytes(kMinQK, 3, 2, 1) <= kMaxSmemPerBlock ? 2 : 1;
  static constexpr int NSTG = kSepStage ? 1 : 0;
  static constexpr int pick_nqk() {
    int n = 6;
    while (n > H && bytes(n, n, NSB, NSTG) > kMaxSmemPerBlock) --n;
    return n;
  }
  static constexpr int NQK = pick_nqk();
  static constexpr int pick_nv() {
    int v = NQK;
    while (!(SO && H == 1) && v < 8 && bytes(NQK, v + 1, NSB, NSTG) <= kMaxSmemPerBlock) ++v;
    return v;
  }
  static constexpr int NV = pick_nv();
  static_assert(NQK >= H && bytes(NQK, NV, NSB, NSTG) <= kMaxSmemPerBlock, "shared memory");
  static constexpr int oV = NQK * kQK;
  static constexpr int oSb = oV + NV * kV;
  static constexpr int oStg = oSb + NSB * kSb;
  static constexpr int oPw = oStg + NSTG * kStg;
  static constexpr int oBar = oPw + kPw;
  static constexpr int oSlot = oBar + kBarBytes;
  static constexpr int oAbort = oSlot + 4;
  static constexpr int oCState = oSlot + 8;  // final c of the rescaled state (float)
  static constexpr int kAlloc = bytes(NQK, NV, NSB, NSTG);
  static_assert(kQK % 1024 == 0 && kV % 1024 == 0 && kSb % 1024 == 0, "align");
  // state_out is staged through the (then idle) rings: rows of DVT + 4 floats
  static constexpr int kStageRow = DVT + 4;
  static_assert(SO || H * 128 * kStageRow * 4 <= kAlloc, "state_out staging");
  // tensor memory: state halves, P buffers, output buffers
  static constexpr int kSCols = H * DVT;
  // Where only one of them fits twice, two O buffers (the outputs of chunk i
  // are read while chunk i+1's products accumulate) measured better than two
  // P buffers (long: 138 us against 142 us).
  static constexpr int NO = (!SO && kSCols + C + 2 * DVT <= 512) ? 2 : 1;
  static constexpr int NP = (!SO && kSCols + 2 * C + NO * DVT <= 512) ? 2 : 1;
  static constexpr int cS = 0, cP = kSCols, cO = kSCols + NP * C;
  static constexpr int kColsUsed = SO ? kSCols : cO + NO * DVT;
  static_assert(kColsUsed <= 512, "tmem");
  static constexpr int kTmemCols = kColsUsed <= 32 ? 32 : kColsUsed <= 64 ? 64 : kColsUsed <= 128 ? 128
                                   : kColsUsed <= 256 ? 256 : 512;
  // The output group handles P of chunk i+1 before the outputs of chunk i when
  // both chunks' Q/K halves and P buffers fit at once and the V ring (whose
  // slots also stage the outputs) is deep enough that chunk i+1's loads do not
  // wait for the store of chunk i-1.
  static constexpr bool kLookahead = !SO && NQK >= 2 * H && NP >= 2 && NO >= 2 && NV >= 3;
  // Completions that coincide share one barrier: P-buffer reuse and (with two
  // or more single-half snapshot buffers) snapshot reuse wait for the output
  // barrier of the chunk that last used the buffer, which implies both.
  static constexpr bool kMergePFree = NP == NO;
  static constexpr bool kMergeSbFree = H == 1 && NSB >= 2 && NSB == NO;
  // State-only pass: one release per chunk frees its K and V slots together.
  static constexpr bool kUnifiedStage = SO && H == 1 && NQK == NV;
  // barriers
  static constexpr int bQkFull = 0, bQkEmpty = NQK, bVFull = 2 * NQK, bVEmpty = 2 * NQK + NV,
                       bWReady = 2 * NQK + 2 * NV, bSRead = 2 * NQK + 3 * NV, bSFull = bSRead + H,
                       bSbReady = bSFull + H, bSbFree = bSbReady + NSB, bPFull = bSbFree + NSB,
                       bPFree = bPFull + NP, bPtReady = bPFree + NP, bOFull = bPtReady + NP,
                       bOFree = bOFull + NO, bFin = bOFree + NO, bSDone = bFin + 1, bNever = bSDone + NV,
                       bQkRot = bNever + 1, kBars = bQkRot + NQK;
  static_assert(kBars * 8 <= kBarBytes, "barriers");
};

struct TcParams {
  const float* gamma;
  const float* state_in;  // state before the first token, [B*H][DK][dv] (null: zero)
  float* state_out;  // main pass: final state (may be null)
  float* ws;         // segment states [B*H][segments-1][DK][dv]
  const float* norm_w;  // GroupNorm of the outputs (NORM kernels): weight, bias [H dv]
  const float* norm_b;  //   (null: one, zero) and eps
  float norm_eps;
  int H, N, dv, n_dv_tiles, BH, segments, seg_chunks, n_chunks;
  int full_units;    // leading units (b*H+h)*n_dv_tiles + tile run whole; the others in `segments`
  int dk;            // query/key width (<= DK; the columns past it are zero-filled by the loads)
  float scale;       // factor of the query (1/sqrt(dk) unless the caller sets another)
  unsigned int test_stall_us;  // > 0: failure-path test (see retention_test_stall_waits)
  const float* theta;  // rotation kernels: frequencies [dk/2] of the position phase rotation
  int n0;              //   and the position of token 0
};

// Position of this CTA.  Units u = (b*H+h) * n_dv_tiles + value tile.  The
// main pass runs units 0 .. full_units-1 whole (CTA u), then the cut units
// segment by segment (segment 0 of each, then segment 1, ...); the pre-pass
// runs segments 0 .. segments-2 of the cut units in the same order.
struct CtaPos {
  int dvt, bh, seg;
  int nseg;        // segments of this unit (1: whole)
  int seg_chunks;  // chunks per segment of this unit
  int cut;         // index of the unit among the cut ones (workspace block), -1 if whole
};
template <bool SO>
__device__ __forceinline__ CtaPos cta_pos(const TcParams& p) {
  const int x = blockIdx.x;
  int u, seg = 0, cut = -1;
  if (!SO && x < p.full_units) {
    u = x;
  } else {
    const int n_cut = p.BH * p.n_dv_tiles - p.full_units;
    const int y = SO ? x : x - p.full_units;
    cut = y % n_cut;
    seg = y / n_cut;
    u = p.full_units + cut;
  }
  const bool whole = cut < 0;
  return CtaPos{u % p.n_dv_tiles, u / p.n_dv_tiles, seg, whole ? 1 : p.segments,
                whole ? p.n_chunks : p.seg_chunks, cut};
}

__device__ __forceinline__ float gamma_pow(float g, float lg, float d) {
  if (d == 0.0f) return 1.0f;
  if (g <= 0.0f) return 0.0f;
  return exp2f(d * lg);
}

// One chunk of the rescaled state's bookkeeping: from c (in [1, 2)) and
// inv_gL = 1 / gamma^L <= 2^14, n = floor(log2(c inv_gL)) in [0, 15] and
// c <- 2^-n c inv_gL.  Any consistent value of c is exact for the method (it
// only rescales the stored state); every thread that needs c or n runs the
// same sequence of these steps, so all of them hold identical values.
__device__ __forceinline__ void frame_advance(float& c, int& n, float inv_gL) {
  const float y = c * inv_gL;
  int e = (int)((__float_as_uint(y) >> 23) & 0xffu) - 127;
  e = e < 0 ? 0 : (e > 15 ? 15 : e);
  n = e;
  c = y * __uint_as_float((uint32_t)(127 - e) << 23);
}

__device__ __forceinline__ void flag_timeout(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_device_status, RET_DEV_WAIT_TIMEOUT);
}

// The waiting loop of wait_bar (limit_ns: how long before it gives up).
__device__ __forceinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      flag_timeout(abort_flag);
      return false;
    }
  }
}

// Wait for phase `parity` of `bar`; false if this CTA is aborting or the wait timed out.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_test_wait(bar, parity)) return true;  // cheap check first (no suspend)
  return wait_bar_slow(bar, parity, abort_flag);
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

// Group-wide wait: every thread of an epilogue group waits, then all agree
// (one barrier with an OR) on whether to go on, so the warps never diverge.
__device__ __forceinline__ bool group_wait(uint32_t id, uint32_t bar, uint32_t parity,
                                           volatile int* abort_flag) {
  const bool ok = wait_bar(bar, parity, abort_flag);
  return !named_bar_or(id, kGroup, !ok || *abort_flag);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Columns col0..col0+31 (col0 % 32 == 0) of row `row`, as 16 packed bf16
// pairs, into a 128-byte-swizzled tile made of 64-column blocks of
// `rows_per_block` rows (the layout of a TMA SWIZZLE_128B box).
__device__ __forceinline__ void store_row32_packed(uint8_t* tile, int rows_per_block, int row,
                                                   int col0, const uint32_t* pk) {
  uint8_t* blk = tile + (col0 / 64) * rows_per_block * 128;
  const int c16 = (col0 % 64) / 8;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(blk + swz128(row, c16 + j)) =
        make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
}

// Slot and phase parity of the next use of an N-slot ring, advanced by one.
template <int N>
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++slot == N) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Descriptor of `addr` + `bytes`: the start address sits in the low 14 bits of
// a shared-memory descriptor in 16-byte units, and shared addresses stay below
// 256 KB, so a byte offset is added to the descriptor directly.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// Byte offset of K-step kk (16 elements) in a K-major, 128-byte-swizzled
// operand of `rows` rows stored as 64-column boxes.
__device__ __forceinline__ uint32_t kmajor_step(int kk, int rows) { return (kk >> 2) * rows * 128 + (kk & 3) * 32; }

// D (+)= A B^T over `steps` K-steps of 16, operands from shared memory; a K-step
// advances A by a_step(kk) and B by b_step(kk) bytes (descriptors are offset,
// not rebuilt, per step).
template <class FA, class FB>
__device__ __forceinline__ void mma_run(uint32_t d, uint64_t da, uint64_t db, uint32_t idesc, int steps,
                                        bool accumulate_first, FA a_step, FB b_step) {
  mma_bf16(d, da, db, idesc, accumulate_first ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < steps; ++kk) mma_bf16(d, desc_add(da, a_step(kk)), desc_add(db, b_step(kk)), idesc, 1u);
}

// Multiply, in place, every bf16 element of row r of a tile of 128-byte rows
// (ROWS rows per 64-column box, NBYTES in total) by f(r).  Each of the group's
// threads loads a batch of up to eight 16-byte units before it scales and
// stores any, so a batch costs about one shared-memory round trip.
template <int NBYTES, int ROWS, class F>
__device__ __forceinline__ void scale_rows_bf16(uint8_t* base, int tid, F f) {
  static_assert(NBYTES % (16 * kGroup) == 0, "tile size");
  constexpr int kUnits = NBYTES / (16 * kGroup);
  constexpr int kBatch = kUnits < 8 ? kUnits : 8;  // at most 32 registers of data in flight
  static_assert(kUnits % kBatch == 0, "batch");
#pragma unroll 1
  for (int k0 = 0; k0 < kUnits; k0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) v[k] = *reinterpret_cast<const uint4*>(base + (tid + (k0 + k) * kGroup) * 16);
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int row = (((tid + (k0 + k) * kGroup) * 16) % (ROWS * 128)) / 128;
      const float s = f(row);
      uint32_t* w = reinterpret_cast<uint32_t*>(&v[k]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 t = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w[j]));
        w[j] = pack_bf16(t.x * s, t.y * s);
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) *reinterpret_cast<uint4*>(base + (tid + (k0 + k) * kGroup) * 16) = v[k];
  }
}

// Final state of a CTA's run of chunks, S^ / c, after every MMA has completed:
// lane-major into the workspace (pre-pass), or row-major into state_out (last
// segment of the main pass) through the then idle shared-memory rings, so the
// global stores are coalesced.  Kept out of line: everything it needs is
// recomputed from the launch parameters, so no register stays live across the
// roles for it.
template <int C, int DK, int DVT, bool SO>
__device__ __noinline__ void write_final_state(const TcParams& p, uint8_t* sm, uint32_t tmem) {
  using L = Cfg<C, DK, DVT, SO>;
  constexpr int H = L::H;
  const CtaPos pos = cta_pos<SO>(p);
  const int dvt = pos.dvt, bh = pos.bh, seg = pos.seg;
  const int nck = min(seg * pos.seg_chunks + pos.seg_chunks, p.n_chunks) - seg * pos.seg_chunks;
  const bool to_out = !SO && seg == pos.nseg - 1 && p.state_out != nullptr;
  if (!(SO || to_out) || nck <= 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dv0 = dvt * DVT;
  if (warp >= 2 && warp < 6) {
    const int quarter = warp & 3;
    const uint32_t lane_addr = (uint32_t)(32 * quarter) << 16;
    const int srow = 32 * quarter + lane;
    const float inv_c = 1.f / *reinterpret_cast<const float*>(sm + L::oCState);
#pragma unroll 1
    for (int hh = 0; hh < H; ++hh) {
#pragma unroll 1
      for (int cb = 0; cb < DVT / 32; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_addr + L::cS + hh * DVT + cb * 32, r);
        tmem_wait_ld();
        float4* dst;
        size_t stride;
        if (SO) {
          // float4 number (c4 * 128 + row) of block (cut unit, segment, half)
          dst = reinterpret_cast<float4*>(p.ws) +
                (((size_t)pos.cut * (p.segments - 1) + seg) * H + hh) * (size_t)(DVT / 4) * 128 +
                (size_t)(cb * 8) * 128 + srow;
          stride = 128;
        } else {
          dst = reinterpret_cast<float4*>(sm) + ((size_t)(hh * 128 + srow) * L::kStageRow) / 4 + cb * 8;
          stride = 1;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j * stride] = make_float4(__uint_as_float(r[4 * j]) * inv_c, __uint_as_float(r[4 * j + 1]) * inv_c,
                                        __uint_as_float(r[4 * j + 2]) * inv_c, __uint_as_float(r[4 * j + 3]) * inv_c);
      }
    }
  }
  if (to_out) {
    __syncthreads();
    const float4* src = reinterpret_cast<const float4*>(sm);
    float* base = p.state_out + (size_t)bh * p.dk * p.dv + dv0;
    const int cols4 = min(DVT, p.dv - dv0) / 4;  // value columns of this tile inside dv
    for (int q4 = threadIdx.x; q4 < p.dk * cols4; q4 += blockDim.x) {
      const int row = q4 / cols4, c4 = q4 % cols4;
      *reinterpret_cast<float4*>(base + (size_t)row * p.dv + 4 * c4) = src[row * (L::kStageRow / 4) + c4];
    }
  }
}

// What the roles of one CTA share, set up by the kernel before they start.
struct RoleCtx {
  const CUtensorMap *tmq, *tmk, *tmv, *tmo;
  uint8_t* sm;
  uint32_t tmem;
  float inv_gC;  // 1 / gamma^C (rescaled form only)
  int pre;       // leading chunks whose loads the set-up already issued
};

// TMA loads of chunk i into the ring slots of layout L: the V slab into V slot
// i % NV, and Q/K half hh into Q/K slot (i H + hh) % NQK.  The caller has made
// sure the slots are free.
template <class L, bool SO>
__device__ __forceinline__ void load_v(uint32_t sbase, const CUtensorMap* tmv, int i, int row, int dv0, int bh) {
  const int s = i % L::NV;
  const uint32_t full = sbase + L::oBar + 8 * (L::bVFull + s), dst = sbase + L::oV + s * L::kV;
  mbar_arrive_expect_tx(full, L::kV);
#pragma unroll
  for (int b = 0; b < L::kDVT / 64; ++b) tma_load_3d(dst + b * L::kC * 128, tmv, dv0 + b * 64, row, bh, full);
}
template <class L, bool SO>
__device__ __forceinline__ void load_qk(uint32_t sbase, const CUtensorMap* tmq, const CUtensorMap* tmk, int u, int hh,
                                        int row, int bh) {
  const int s = u % L::NQK;
  const uint32_t full = sbase + L::oBar + 8 * (L::bQkFull + s), dst = sbase + s * L::kQK;
  mbar_arrive_expect_tx(full, L::kQK);
  if (!SO) {
#pragma unroll
    for (int b = 0; b < 2; ++b) tma_load_3d(dst + b * L::kC * 128, tmq, hh * 128 + b * 64, row, bh, full);
  }
#pragma unroll
  for (int b = 0; b < 2; ++b) tma_load_3d(dst + L::kQ + b * L::kC * 128, tmk, hh * 128 + b * 64, row, bh, full);
}

// The four roles of a CTA (producer, MMA issuer, state group, output group).
// FAST selects the rescaled form; a CTA picks one instantiation at its start,
// so the code it runs holds no branches of the other form.
template <int C, int DK, int DVT, bool SO, bool FAST, bool NORM, bool ROT, bool REV>
__device__ __forceinline__ void chunk_roles(const TcParams& p, const RoleCtx& x) {
  using L = Cfg<C, DK, DVT, SO>;
  constexpr int H = L::H, NQK = L::NQK, NV = L::NV, NP = L::NP, NO = L::NO, NSB = L::NSB;
  constexpr bool fast = FAST;
  constexpr bool look = L::kLookahead;
  uint8_t* sm = x.sm;
  const uint32_t sbase = smem_u32(sm);
  const uint32_t tmem = x.tmem;
  const float inv_gC = x.inv_gC;
  float* pw = reinterpret_cast<float*>(sm + L::oPw);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::oAbort);
  auto bar = [&](int i) { return sbase + L::oBar + 8 * i; };
  auto qk_q = [&](int s) { return sbase + s * L::kQK; };
  auto qk_k = [&](int s) { return sbase + s * L::kQK + L::kQ; };
  auto v_slot = [&](int s) { return sbase + L::oV + s * L::kV; };
  auto sb_buf = [&](int b) { return sbase + L::oSb + b * L::kSb; };
  const CtaPos pos = cta_pos<SO>(p);
  const int dvt = pos.dvt, bh = pos.bh, seg = pos.seg;
  const int head = bh % p.H;
  const int c_begin = seg * pos.seg_chunks;
  const int nck = min(c_begin + pos.seg_chunks, p.n_chunks) - c_begin;
  const int dv0 = dvt * DVT;
  // Time reversed (rev): chunks are taken from the last to the first, and in
  // a chunk of len tokens row r plays the part of row len-1-r of the causal
  // form: in-chunk weights gamma^(c-r) for keys c >= r, gamma^(len-r) on the
  // incoming state, gamma^r on the state update.
  constexpr bool rev = REV;
  static_assert(!(REV && (NORM || ROT)), "time reversal without GroupNorm or the rotation");
  const float g = p.gamma[head];
  const float lg = g > 0.f ? log2f(g) : 0.f;
  const bool zero_init = SO || (seg == 0 && p.state_in == nullptr);
  // The state-only pass walks its segment from the last chunk back to the
  // first (its sum does not depend on the order; the weights then need no
  // running rescale).  chunk_at(i) is the sequence chunk of the CTA's i-th step.
  auto chunk_at = [&](int i) {
    const int j = SO ? c_begin + nck - 1 - i : c_begin + i;
    return rev ? p.n_chunks - 1 - j : j;
  };
  auto chunk_len = [&](int i) { return min(C, p.N - chunk_at(i) * C); };
  // Segment states in the workspace are stored lane-major: float4 number
  // (c4 * 128 + row) of block (cut unit, segment, half) holds columns
  // 4c4..4c4+3 of state row `row`, so a warp's 32 rows are 512 contiguous bytes.
  auto ws_block = [&](int s, int hh) {
    return reinterpret_cast<float4*>(p.ws) + (((size_t)pos.cut * (p.segments - 1) + s) * H + hh) * (size_t)(DVT / 4) * 128;
  };
  auto inv_g = [&](int i) {
    const int len = chunk_len(i);
    return len == C ? inv_gC : 1.f / pw[len];
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Initial state of a segment that does not start from zero: the caller's
  // state, decayed to the segment's first token, plus the decayed sum of the
  // preceding segments' local end states (written by the pre-pass); state
  // row `srow`, 32-column blocks cb0..cb1-1 of each half, into the state
  // columns.  The state and output groups each take half the columns (the
  // blocks are L2 hits, so latency sets the cost: more threads, more loads in
  // flight), then meet at a barrier of both groups.
  auto init_state = [&](int srow, uint32_t lane_addr, int cb0, int cb1) {
    if (seg > 0) griddep_wait();  // the pre-pass wrote the workspace
    const float seg_len = (float)pos.seg_chunks * (float)C;
    // time reversed: the first segment holds the short chunk, so the caller's
    // state (after the last token) is pad tokens closer to later segments
    const float pad = rev && seg > 0 ? (float)(p.n_chunks * C - p.N) : 0.f;
#pragma unroll 1
    for (int hh = 0; hh < H; ++hh) {
#pragma unroll 1
      for (int cb = cb0; cb < cb1; ++cb) {
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0.f;
        const int row = hh * 128 + srow;
        if (p.state_in != nullptr && row < p.dk) {
          // gamma^(seg Lseg) state_in, row hh*128 + srow, columns dv0 + 32 cb ..
          // (rows past dk and columns past dv are padding: they stay zero)
          const float f = gamma_pow(g, lg, (float)seg * seg_len - pad);
          const int col = dv0 + cb * 32;
          const float4* src = reinterpret_cast<const float4*>(p.state_in + ((size_t)bh * p.dk + row) * p.dv + col);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 x = col + 4 * j < p.dv ? __ldg(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            acc[4 * j + 0] = f * x.x;
            acc[4 * j + 1] = f * x.y;
            acc[4 * j + 2] = f * x.z;
            acc[4 * j + 3] = f * x.w;
          }
        }
        // three segments' loads in flight per round trip
#pragma unroll 1
        for (int t0 = 0; t0 < seg; t0 += 3) {
          float4 x[3][8];
#pragma unroll
          for (int tt = 0; tt < 3; ++tt) {
            if (t0 + tt < seg) {
              const float4* src = ws_block(t0 + tt, hh) + (size_t)(cb * 8) * 128 + srow;
#pragma unroll
              for (int j = 0; j < 8; ++j) x[tt][j] = __ldcg(src + j * 128);
            }
          }
#pragma unroll
          for (int tt = 0; tt < 3; ++tt) {
            if (t0 + tt < seg) {
              const float f = gamma_pow(g, lg, (float)(seg - 1 - t0 - tt) * seg_len);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                acc[4 * j + 0] = fmaf(f, x[tt][j].x, acc[4 * j + 0]);
                acc[4 * j + 1] = fmaf(f, x[tt][j].y, acc[4 * j + 1]);
                acc[4 * j + 2] = fmaf(f, x[tt][j].z, acc[4 * j + 2]);
                acc[4 * j + 3] = fmaf(f, x[tt][j].w, acc[4 * j + 3]);
              }
            }
          }
        }
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(acc[j]);
        tmem_st32(tmem + lane_addr + L::cS + hh * DVT + cb * 32, r);
      }
    }
    tmem_wait_st();
    tc_fence_before();  // the other group reads these columns next
    named_bar_sync(kBarInit, 2 * kGroup);
    tc_fence_after();
  };

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      // the set-up issued the loads of the first x.pre chunks
      int v_issued = x.pre, qk_issued = x.pre * H;
      bool ok = true;
      for (int i = x.pre; i < nck && ok; ++i) {
        const int row = chunk_at(i) * C;
        {
          const int s = i % NV, k = i / NV;
          if (k > 0 && !wait_bar(bar(L::bVEmpty + s), (k - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          load_v<L, SO>(sbase, x.tmv, i, row, dv0, bh);
          v_issued = i + 1;
        }
        for (int hh = 0; hh < H; ++hh) {
          const int u = i * H + hh, s = u % NQK, k = u / NQK;
          if (!L::kUnifiedStage && k > 0 && !wait_bar(bar(L::bQkEmpty + s), (k - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          load_qk<L, SO>(sbase, x.tmq, x.tmk, u, hh, row, bh);
          qk_issued = u + 1;
        }
      }
      // every issued load has landed before the CTA may exit
      for (int i = v_issued - 1; i >= 0 && i >= v_issued - NV; --i)
        drain_bar(bar(L::bVFull + i % NV), (i / NV) & 1, abort_flag);
      for (int u = qk_issued - 1; u >= 0 && u >= qk_issued - NQK; --u)
        drain_bar(bar(L::bQkFull + u % NQK), (u / NQK) & 1, abort_flag);
    }
  } else if (warp == 1 || warp == kIssuerWarpB) {
    // ================= MMA issuers =================
    // Two threads issue the MMAs, each a chain of dependent instructions
    // (waits, bookkeeping, MMAs): lane 0 of warp 1 (A) issues Q K^T and the
    // state update, lane 0 of warp kIssuerWarpB (B) the two products that
    // accumulate into O, Q S and P~ W, so the O accumulator keeps one issue
    // order.  The state-only pass has A alone.  Slots both read are freed
    // by a commit from each; B issues P~ W(i) only after the state update of
    // chunk i (which also reads W) has completed, so its release of the V
    // slot (or the output group's, when outputs are staged in the slot)
    // covers A's read too.  Ring slots and parities are running counters and
    // operand descriptors a per-ring base plus slot stride.
    if (lane == 0 && (warp == 1 || !SO)) {
      constexpr uint32_t idP = make_idesc(C, C, false, false);
      constexpr uint32_t idO = make_idesc(C, DVT, false, true);
      constexpr uint32_t idS = make_idesc(128, DVT, true, true);
      constexpr uint32_t kQKs = L::kQK >> 4, kVs = L::kV >> 4, kSbs = L::kSb >> 4;  // slot strides
      const uint64_t dQ = make_sdesc(qk_q(0), 16, 1024);          // Q, K-major A (Q K^T, Q S)
      const uint64_t dKb = make_sdesc(qk_k(0), 16, 1024);         // K, K-major B (Q K^T)
      const uint64_t dKa = make_sdesc(qk_k(0), C * 128, 1024);    // K^T, MN-major A (state)
      const uint64_t dV = make_sdesc(v_slot(0), C * 128, 1024);   // W or V, MN-major B
      const uint64_t dSb = make_sdesc(sb_buf(0), 128 * 128, 1024);  // snapshot, MN-major B
      // Q/K slots are ready once loaded, or, with the rotation group, once turned
      const uint32_t bQkFull = bar(ROT ? L::bQkRot : L::bQkFull), bQkEmpty = bar(L::bQkEmpty), bVFull = bar(L::bVFull),
                     bVEmpty = bar(L::bVEmpty), bWReady = bar(L::bWReady), bSRead = bar(L::bSRead),
                     bSFull = bar(L::bSFull), bSbReady = bar(L::bSbReady), bSbFree = bar(L::bSbFree),
                     bPFull = bar(L::bPFull), bPFree = bar(L::kMergePFree ? L::bOFull : L::bPFree),
                     bPtReady = bar(L::bPtReady), bOFull = bar(L::bOFull), bOFree = bar(L::bOFree),
                     bSDone = bar(L::bSDone);
      auto wait = [&](uint32_t b, uint32_t par) { return wait_bar(b, par & 1u, abort_flag); };
      auto has_state = [&](int i) { return i > 0 || !zero_init; };
      bool ok = true;
      if (warp == 1) {
        // ---------- issuer A: Q K^T and the state update ----------
        // state update of one half: S_h = 2^-n S_h + K_h^T W (S_h = K_h^T W when the state is zero)
        auto mma_s = [&](uint32_t d, int qslot, int vslot, bool hs, int n) {
          const uint64_t a = dKa + (uint64_t)qslot * kQKs, b = dV + (uint64_t)vslot * kVs;
          if (hs) mma_bf16_scaled(d, a, b, idS, n);
          else mma_bf16(d, a, b, idS, 0u);
#pragma unroll
          for (int kk = 1; kk < C / 16; ++kk) mma_bf16(d, a + kk * 128, b + kk * 128, idS, 1u);
        };
        float c = 1.f;
        int n = 0;
        RingPos<NQK> qk_w;  // next Q/K unit to wait for
        int qk_waited = 0;
        auto wait_qk = [&](int u_end) -> bool {
          while (qk_waited < u_end) {
            if (!wait(bQkFull + 8 * qk_w.slot, qk_w.phase)) return false;
            qk_w.next();
            ++qk_waited;
          }
          return true;
        };
        if (SO) {
          // state only, last chunk first: S += K^T W with every chunk's decay
          // in its W (any gamma), one accumulating MMA chain
          RingPos<NV> v;
          RingPos<NQK> qs;
          for (int i = 0; i < nck && ok; ++i) {
            if (!wait(bWReady + 8 * v.slot, v.phase)) {
              ok = false;
              break;
            }
            for (int hh = 0; hh < H && ok; ++hh) {
              ok = wait_qk(i * H + hh + 1);
              if (!ok) break;
              tc_fence_after();
              mma_s(tmem + L::cS + hh * DVT, qs.slot, v.slot, i > 0, 0);
              if (!L::kUnifiedStage) mma_commit(bQkEmpty + 8 * qs.slot);
              qs.next();
            }
            if (ok) mma_commit(bVEmpty + 8 * v.slot);
            v.next();
          }
        } else {
          // With lookahead (chunk i+1's Q K^T may run while chunk i still
          // holds its P buffer) chunk i issues S(i), Q K^T(i+1); without,
          // Q K^T(i), S(i).
          RingPos<NQK> q_p, q_s;  // Q/K slot of the next unit for Q K^T, and for S
          RingPos<NV> v_s;        // V slot of the next chunk for S
          // P[j % NP] = Q_j K_j^T
          auto issue_p = [&](int j) -> bool {
            const int pb = j & (NP - 1);
            if (j >= NP && !wait(bPFree + 8 * pb, (uint32_t)(j / NP - 1))) return false;
            if (!wait_qk((j + 1) * H)) return false;
            tc_fence_after();
#pragma unroll 1
            for (int hh = 0; hh < H; ++hh) {
              const uint64_t a = dQ + (uint64_t)q_p.slot * kQKs, b = dKb + (uint64_t)q_p.slot * kQKs;
              q_p.next();
              mma_run(tmem + L::cP + pb * C, a, b, idP, 8, hh > 0, [](int kk) { return kmajor_step(kk, C); },
                      [](int kk) { return kmajor_step(kk, C); });
            }
            mma_commit(bPFull + 8 * pb);
            return true;
          };
          // state update of chunk i, half by half
          auto issue_s = [&](int i) -> bool {
            if (!wait(bWReady + 8 * v_s.slot, v_s.phase)) return false;
            if (!fast && !wait(bVFull + 8 * v_s.slot, v_s.phase)) return false;
            if (fast) frame_advance(c, n, inv_g(i));
            for (int hh = 0; hh < H; ++hh) {
              if (!wait_qk(i * H + hh + 1) || !wait(bSRead + 8 * hh, (uint32_t)i)) return false;
              tc_fence_after();
              mma_s(tmem + L::cS + hh * DVT, q_s.slot, v_s.slot, has_state(i), fast ? n : 0);
              mma_commit(bSFull + 8 * hh);
              mma_commit(bQkEmpty + 8 * q_s.slot);  // A's reads of the Q/K half are done
              q_s.next();
            }
            mma_commit(bSDone + 8 * v_s.slot);  // W of this V slot is no longer read by A
            v_s.next();
            return true;
          };
          // one call site per step keeps the issuer's code small
          if (look) {
            for (int i = -1; i < nck && ok; ++i) {
              if (i >= 0) ok = issue_s(i);
              if (ok && i + 1 < nck) ok = issue_p(i + 1);
            }
          } else {
            for (int i = 0; i < nck && ok; ++i) ok = issue_p(i) && issue_s(i);
          }
        }
      } else {
        // ---------- issuer B: O (+)= Q S, then O += P~ W ----------
        RingPos<NQK> q_b;  // Q/K slot of the next unit for Q S
        RingPos<NV> v_b;   // V slot of the next chunk
        for (int i = 0; i < nck && ok; ++i) {
          const int ob = i & (NO - 1), pb = i & (NP - 1);
          // W (and, in the direct form, the scaled Q) of chunk i, and a free O buffer
          ok = wait(bWReady + 8 * v_b.slot, v_b.phase) && (i < NO || wait(bOFree + 8 * ob, (uint32_t)(i / NO - 1)));
          for (int hh = 0; hh < H && ok; ++hh) {
            const int u = i * H + hh, b = u & (NSB - 1);
            ok = wait(bQkFull + 8 * q_b.slot, q_b.phase) && wait(bSbReady + 8 * b, (uint32_t)(u / NSB));
            if (!ok) break;
            tc_fence_after();
            if (has_state(i))
              mma_run(tmem + L::cO + ob * DVT, dQ + (uint64_t)q_b.slot * kQKs, dSb + (uint64_t)b * kSbs, idO, 8,
                      hh > 0, [](int kk) { return kmajor_step(kk, C); }, [](int kk) { return (uint32_t)kk * 2048; });
            if (!L::kMergeSbFree) mma_commit(bSbFree + 8 * b);
            mma_commit(bQkEmpty + 8 * q_b.slot);  // B's read of the Q half is done
            q_b.next();
          }
          // P~ of chunk i, and its state update done with W
          ok = ok && wait(bPtReady + 8 * pb, (uint32_t)(i / NP)) && wait(bSDone + 8 * v_b.slot, v_b.phase);
          if (!ok) break;
          tc_fence_after();
          const uint64_t db = dV + (uint64_t)v_b.slot * kVs;
          const uint32_t dO = tmem + L::cO + ob * DVT, aP = tmem + L::cP + pb * C;
          mma_bf16_ta(dO, aP, db, idO, has_state(i) ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < C / 16; ++kk) mma_bf16_ta(dO, aP + kk * 8, db + kk * 128, idO, 1u);
          mma_commit(bOFull + 8 * ob);
          if (!L::kMergePFree) mma_commit(bPFree + 8 * pb);
          if (L::kSepStage) mma_commit(bVEmpty + 8 * v_b.slot);  // V slot free once the MMAs are done
          v_b.next();
        }
      }
      // every MMA either thread issued has completed before TMEM is released
      mma_commit(bar(L::bFin));
      if (warp == 1) drain_bar(bar(L::bFin), 0, abort_flag);
    }
  } else if (warp < 6) {
    // ================= state group (warps 2..5) =================
    const int et = threadIdx.x - 64;
    const int quarter = warp & 3;
    const uint32_t lane_addr = (uint32_t)(32 * quarter) << 16;
    const int srow = 32 * quarter + lane;  // state row inside a 128-row half
    // The group's waits are per warp (all lanes agree): the state group has no
    // barrier of its own, so a warp that gives up strands no other, and no
    // warp waits for the slowest of the four at every step.
    auto gw = [&](int b, uint32_t par) {
      const bool ok = wait_bar(bar(b), par & 1u, abort_flag);
      return __all_sync(0xffffffffu, ok && !*abort_flag);
    };

    if (!zero_init) init_state(srow, lane_addr, 0, DVT / 64);

    // W = diag(c gamma^(L-1-m)) V, in place in the chunk's V slot
    auto w_pass = [&](int i, float ci) -> bool {
      const int vs = i % NV;
      if (!gw(L::bVFull + vs, (i / NV) & 1)) return false;
      const int len = chunk_len(i);
      scale_rows_bf16<L::kV, C>(sm + L::oV + vs * L::kV, et,
                                [&](int r) { return r < len ? ci * pw[rev ? r : len - 1 - r] : 0.f; });
      fence_proxy_async_smem();
      mbar_arrive(bar(L::bWReady + vs));
      return true;
    };
    // direct form: K <- diag(gamma^(L-1-m)) K and Q <- diag(scale gamma^(t+1)) Q in place
    auto kq_pass = [&](int i) -> bool {
      const int len = chunk_len(i);
      if (!gw(L::bPFull + i % NP, (i / NP) & 1)) return false;
      for (int hh = 0; hh < H; ++hh) {
        const int s = (i * H + hh) % NQK;
        scale_rows_bf16<L::kK, C>(sm + s * L::kQK + L::kQ, et,
                                  [&](int r) { return r < len ? pw[rev ? r : len - 1 - r] : 0.f; });
        if (!SO)
          scale_rows_bf16<(SO ? L::kK : L::kQ), C>(
              sm + s * L::kQK, et, [&](int r) { return r < len ? p.scale * pw[rev ? len - r : r + 1] : 0.f; });
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(L::bWReady + i % NV));
      return true;
    };
    // bf16 copy of the state for the Q S product of chunk i (times 2^-n in the
    // rescaled form; the direct form also decays the state by gamma^L here)
    auto snapshot = [&](int i, int n, float gL) -> bool {
      const bool has_state = i > 0 || !zero_init;
#pragma unroll 1
      for (int hh = 0; hh < H; ++hh) {
        const uint32_t tS = tmem + lane_addr + L::cS + hh * DVT;
        const int u = i * H + hh, b = u % NSB;
        uint8_t* sb = sm + L::oSb + b * L::kSb;
        const bool sb_free = u < NSB;  // no earlier Q S product reads this buffer
        auto wait_sb = [&] { return sb_free || gw(L::kMergeSbFree ? L::bOFull + b : L::bSbFree + b, (u / NSB - 1) & 1); };
        const bool whole_row = has_state && fast && DVT == 128;
        if (!whole_row && !wait_sb()) return false;
        if (has_state && i > 0 && !gw(L::bSFull + hh, (i - 1) & 1)) return false;
        if (whole_row) {
          // the whole row in flight at once, so the state MMA is released
          // before any of it is packed, and before the snapshot buffer is free
          tc_fence_after();
          const float f = __uint_as_float((uint32_t)(127 - n) << 23);  // 2^-n
          uint32_t r[128];
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld32p(tS + q * 32, &r[q * 32]);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(L::bSRead + hh));  // the state MMA may overwrite S now
          if (!wait_sb()) return false;
#pragma unroll
          for (int cb = 0; cb < 4; cb += 2) {
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
              pk[j] = pack_bf16(f * __uint_as_float(r[cb * 32 + 2 * j]), f * __uint_as_float(r[cb * 32 + 2 * j + 1]));
            store_row32_packed(sb, 128, srow, cb * 32, &pk[0]);
            store_row32_packed(sb, 128, srow, cb * 32 + 32, &pk[16]);
          }
          fence_proxy_async_smem();
        } else if (has_state) {
          tc_fence_after();
          const float f = fast ? __uint_as_float((uint32_t)(127 - n) << 23) : 1.f;  // 2^-n
#pragma unroll 1
          for (int cb = 0; cb < DVT / 32; cb += 2) {
            uint32_t r[64];
            tmem_ld32p(tS + cb * 32, &r[0]);
            tmem_ld32p(tS + cb * 32 + 32, &r[32]);
            tmem_wait_ld();
            if (!fast) {
              // direct form: decay the state by gamma^L in place
              uint32_t t[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) t[j] = __float_as_uint(__uint_as_float(r[j]) * gL);
              tmem_st32(tS + cb * 32, t);
#pragma unroll
              for (int j = 0; j < 32; ++j) t[j] = __float_as_uint(__uint_as_float(r[32 + j]) * gL);
              tmem_st32(tS + cb * 32 + 32, t);
              if (cb + 2 >= DVT / 32) tmem_wait_st();
            }
            if (cb + 2 >= DVT / 32) {
              tc_fence_before();
              mbar_arrive(bar(L::bSRead + hh));  // the state MMA may overwrite S now
            }
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
              pk[j] = pack_bf16(f * __uint_as_float(r[2 * j]), f * __uint_as_float(r[2 * j + 1]));
            store_row32_packed(sb, 128, srow, cb * 32, &pk[0]);
            store_row32_packed(sb, 128, srow, cb * 32 + 32, &pk[16]);
          }
          fence_proxy_async_smem();
        } else {
          tc_fence_before();
          mbar_arrive(bar(L::bSRead + hh));
        }
        mbar_arrive(bar(L::bSbReady + b));
      }
      return true;
    };

    float c = 1.f;
    int n = 0;
    bool alive = true;
    if (SO) {
      // last chunk first: the i-th step's tokens are weighted by gamma to the
      // number of tokens after them in the segment (c stays 1)
      float after = 0.f;
      for (int i = 0; i < nck && alive; ++i) {
        alive = w_pass(i, gamma_pow(g, lg, after));
        after += (float)chunk_len(i);
      }
    } else {
      if (fast) {
        float c_next = 1.f;
        int n_next = 0;
        for (int i = -1; i < nck && alive; ++i) {
          if (i >= 0) {
            c = c_next;
            n = n_next;
            if (!snapshot(i, n, 1.f)) { alive = false; break; }
          }
          if (i + 1 < nck) {
            frame_advance(c_next, n_next, inv_g(i + 1));
            if (!w_pass(i + 1, c_next)) { alive = false; break; }
          }
        }
      } else {
        for (int i = 0; i < nck && alive; ++i) {
          if (!kq_pass(i)) { alive = false; break; }
          if (!snapshot(i, 0, pw[chunk_len(i)])) { alive = false; break; }
        }
      }
    }
    if (et == 0) *reinterpret_cast<float*>(sm + L::oCState) = c;
  } else {
    // ================= output group (warps 6..9) =================
    const int eo = threadIdx.x - 192;
    const int quarter = warp & 3;
    const uint32_t lane_addr = (uint32_t)(32 * quarter) << 16;
    const int arow = acc_row(C, quarter, lane);  // token row of the C-row accumulators, -1 if none
    if (!SO && !zero_init) init_state(32 * quarter + lane, lane_addr, DVT / 64, DVT / 32);
    auto go = [&](int b, uint32_t par) { return group_wait(kBarO, bar(b), par, abort_flag); };
    bool alive = true;

    // Rotation kernels: the position phase rotation of the queries and keys
    // of each Q/K slot, in place, once the slot has landed and before the MMA
    // issuers read it ("2. Relative Position via Complex Exponential Phase
    // Rotations": pair (2j, 2j+1) of the token at position n0 + n turned by
    // (n0 + n) theta_j).  Thread eo owns the 16-byte unit c16 = eo % 16
    // (pairs 4 c16 .. 4 c16 + 3 of a 128-column half) of rows eo / 16 + 8 m.
    // Per slot it takes the cosine and sine of its first row's angle, reduced
    // modulo 2 pi as in the standalone rotation, and advances them 8 rows at
    // a time by the rotation through 8 theta_j (at most 16 steps, ~1e-7 of
    // rounding each), four rows per batch with every load of a batch issued
    // before any store.  The state-only pass turns keys only.
    RingPos<NQK> qk_rot;
    auto rotate_chunk = [&](int i) -> bool {
      if constexpr (ROT) {
        const int c16 = eo & 15, r0 = eo >> 4;
        constexpr int kStep = kGroup / 16;  // rows between a thread's rows
        constexpr int kRows = 4;            // rows per batch: every load of a batch before any store
        static_assert(C % (kRows * kStep) == 0, "rotation batches");
#pragma unroll 1
        for (int hh = 0; hh < H; ++hh) {
          if (!go(L::bQkFull + qk_rot.slot, qk_rot.phase)) return false;
          uint8_t* qs = sm + qk_rot.slot * L::kQK;
          uint8_t* ks = qs + L::kQ;
          // this half's frequencies and the rotation through kStep rows (kept
          // in registers: arrays shared with the rest of the role would live
          // in memory)
          float tj[4], cj[4], sj[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = hh * 64 + 4 * c16 + e;
            tj[e] = 2 * j < p.dk ? __ldg(p.theta + j) : 0.f;
            const float a = reduced_angle((float)kStep, tj[e]);
            sj[e] = __sinf(a);
            cj[e] = __cosf(a);
          }
          float ca[4], sa[4];
          const float pos = (float)(p.n0 + chunk_at(i) * C + r0);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = reduced_angle(pos, tj[e]);
            sa[e] = __sinf(a);
            ca[e] = __cosf(a);
          }
#pragma unroll 1
          for (int row = r0; row < C; row += kRows * kStep) {
            uint32_t off[kRows];
            uint4 vq[kRows], vk[kRows];
#pragma unroll
            for (int t = 0; t < kRows; ++t) {
              off[t] = (uint32_t)((c16 >> 3) * C * 128) + swz128(row + t * kStep, c16 & 7);
              if (!SO) vq[t] = *reinterpret_cast<const uint4*>(qs + off[t]);
              vk[t] = *reinterpret_cast<const uint4*>(ks + off[t]);
            }
#pragma unroll
            for (int t = 0; t < kRows; ++t) {
              if (!SO)
                vq[t] = make_uint4(rot_pair(vq[t].x, ca[0], sa[0]), rot_pair(vq[t].y, ca[1], sa[1]),
                                   rot_pair(vq[t].z, ca[2], sa[2]), rot_pair(vq[t].w, ca[3], sa[3]));
              vk[t] = make_uint4(rot_pair(vk[t].x, ca[0], sa[0]), rot_pair(vk[t].y, ca[1], sa[1]),
                                 rot_pair(vk[t].z, ca[2], sa[2]), rot_pair(vk[t].w, ca[3], sa[3]));
#pragma unroll
              for (int e = 0; e < 4; ++e) {  // advance kStep rows
                const float cn = ca[e] * cj[e] - sa[e] * sj[e];
                sa[e] = sa[e] * cj[e] + ca[e] * sj[e];
                ca[e] = cn;
              }
            }
#pragma unroll
            for (int t = 0; t < kRows; ++t) {
              if (!SO) *reinterpret_cast<uint4*>(qs + off[t]) = vq[t];
              *reinterpret_cast<uint4*>(ks + off[t]) = vk[t];
            }
          }
          fence_proxy_async_smem();  // the MMAs read the turned pairs through the async proxy
          mbar_arrive(bar(L::bQkRot + qk_rot.slot));
          qk_rot.next();
        }
      }
      return true;
    };
    if constexpr (SO) {
      // state-only pass: this group has nothing else to do
      if constexpr (ROT)
        for (int i = 0; i < nck && alive; ++i) alive = rotate_chunk(i);
    } else {
    if (p.test_stall_us > 0) {
      // Failure-path test: one wait on a barrier nothing completes, with a
      // short limit; it gives up, raises the abort flag and sets the device
      // status bit, and every role unwinds as after a real timeout.
      const bool ok = wait_bar_slow(bar(L::bNever), 0, abort_flag, 1000ull * p.test_stall_us);
      alive = !named_bar_or(kBarO, kGroup, !ok || *abort_flag);
    }

    // P~ = causal mask of P (rescaled form) or (P (.) D) scale (direct form),
    // written as bf16 pairs in place over the first C/2 columns of its buffer
    auto ptilde = [&](int j) -> bool {
      const int pb = j % NP;
      if (!go(L::bPFull + pb, (j / NP) & 1)) return false;
      tc_fence_after();
      const uint32_t tP = tmem + lane_addr + L::cP + pb * C;
#pragma unroll 1
      for (int cb = 0; cb < C / 32; cb += 2) {
        uint32_t r[64];
        tmem_ld32p(tP + cb * 32, &r[0]);
        tmem_ld32p(tP + cb * 32 + 32, &r[32]);
        tmem_wait_ld();
        uint32_t pk[32];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int c0 = cb * 32 + 2 * jj;
          float a = __uint_as_float(r[2 * jj]), b = __uint_as_float(r[2 * jj + 1]);
          // causal: key c <= query row; time reversed: key c >= query row
          const int da = rev ? c0 - arow : arow - c0, db = rev ? c0 + 1 - arow : arow - c0 - 1;
          const bool ka = arow >= 0 && da >= 0, kb = arow >= 0 && db >= 0;
          if (fast) {
            a = ka ? a : 0.f;
            b = kb ? b : 0.f;
          } else {
            a = ka ? pw[da] * p.scale * a : 0.f;
            b = kb ? pw[db] * p.scale * b : 0.f;
          }
          pk[jj] = pack_bf16(a, b);
        }
        // P~ columns 16*cb .. 16*cb+31 lie in P columns already read
        tmem_st16(tP + cb * 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
        tmem_st16(tP + cb * 16 + 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[16]));
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(L::bPtReady + pb));
      return true;
    };
    // out rows = O rows scaled, bf16, staged in the chunk's V slot, TMA-stored
    auto out_chunk = [&](int i, float ci) -> bool {
      const int ob = i % NO;
      if (!go(L::bOFull + ob, (i / NO) & 1)) return false;
      tc_fence_after();
      const int len = chunk_len(i);
      float rt = 0.f;
      if (arow >= 0 && arow < len) rt = fast ? p.scale / (ci * pw[rev ? arow : len - 1 - arow]) : 1.f;
      const int vs = i % NV;
      uint8_t* stg = L::kSepStage ? sm + L::oStg : sm + L::oV + vs * L::kV;
      const uint32_t tO = tmem + lane_addr + L::cO + ob * DVT;
      // GroupNorm of the row (NORM kernels; the row is the head's dv = DVT
      // channels): first pass for its mean and variance, from sums shifted by
      // the row's first value (no cancellation when the mean is large)
      float mu = 0.f, inv = 0.f;
      if constexpr (NORM) {
        float x0 = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll 1
        for (int cb = 0; cb < DVT / 32; cb += 2) {
          uint32_t r[64];
          tmem_ld32p(tO + cb * 32, &r[0]);
          tmem_ld32p(tO + cb * 32 + 32, &r[32]);
          tmem_wait_ld();
          if (cb == 0) x0 = rt * __uint_as_float(r[0]);
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const float d = fmaf(rt, __uint_as_float(r[j]), -x0);
            s1 += d;
            s2 = fmaf(d, d, s2);
          }
        }
        const float m1 = s1 * (1.f / DVT);
        mu = x0 + m1;
        inv = rsqrtf(fmaxf(fmaf(-m1, m1, s2 * (1.f / DVT)), 0.f) + p.norm_eps);
      }
#pragma unroll 1
      for (int cb = 0; cb < DVT / 32; cb += 2) {
        uint32_t r[64];
        tmem_ld32p(tO + cb * 32, &r[0]);
        tmem_ld32p(tO + cb * 32 + 32, &r[32]);
        tmem_wait_ld();
        if (cb + 2 >= DVT / 32) {
          tc_fence_before();
          mbar_arrive(bar(L::bOFree + ob));  // the next product may overwrite O now
        }
        // the staging buffer is free once the previous store has read it: the
        // thread that issued that store waits for this before the barrier
        if (L::kSepStage && cb == 0) {
          if (eo == 0) bulk_wait_group_read0();
          named_bar_sync(kBarO, kGroup);
        }
        if (arow >= 0) {
          uint32_t pk[32];
          if constexpr (NORM) {
            // (o - mu) / sqrt(var + eps) * weight + bias, channel h dv + c
            const int c0 = head * p.dv + cb * 32;
#pragma unroll
            for (int q4 = 0; q4 < 16; ++q4) {
              const float4 w = p.norm_w ? __ldg(reinterpret_cast<const float4*>(p.norm_w + c0) + q4)
                                        : make_float4(1.f, 1.f, 1.f, 1.f);
              const float4 bb = p.norm_b ? __ldg(reinterpret_cast<const float4*>(p.norm_b + c0) + q4)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
              const float y0 = fmaf(fmaf(rt, __uint_as_float(r[4 * q4]), -mu) * inv, w.x, bb.x);
              const float y1 = fmaf(fmaf(rt, __uint_as_float(r[4 * q4 + 1]), -mu) * inv, w.y, bb.y);
              const float y2 = fmaf(fmaf(rt, __uint_as_float(r[4 * q4 + 2]), -mu) * inv, w.z, bb.z);
              const float y3 = fmaf(fmaf(rt, __uint_as_float(r[4 * q4 + 3]), -mu) * inv, w.w, bb.w);
              pk[2 * q4] = pack_bf16(y0, y1);
              pk[2 * q4 + 1] = pack_bf16(y2, y3);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              pk[j] = pack_bf16(rt * __uint_as_float(r[2 * j]), rt * __uint_as_float(r[2 * j + 1]));
          }
          store_row32_packed(stg, C, arow, cb * 32, &pk[0]);
          store_row32_packed(stg, C, arow, cb * 32 + 32, &pk[16]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(kBarO, kGroup);
      if (eo == 0) {
        const int row0 = chunk_at(i) * C;
#pragma unroll
        for (int b = 0; b < DVT / 64; ++b) {
          if constexpr (NORM)  // [B][N][H][dv]: (channel, head, token, batch row)
            tma_store_4d(x.tmo, smem_u32(stg) + b * C * 128, dv0 + b * 64, head, row0, bh / p.H);
          else
            tma_store_3d(x.tmo, smem_u32(stg) + b * C * 128, dv0 + b * 64, row0, bh);
        }
        bulk_commit_group();
        if (!L::kSepStage) {
          bulk_wait_group_read0();  // the V slot may be reloaded once the store has read it
          mbar_arrive(bar(L::bVEmpty + vs));
        }
      }
      return true;
    };

    float c = 1.f;
    int n = 0;
    // Rotation kernels.  With lookahead, chunks 0 and 1 are turned first and
    // chunk i+2 between the mask of chunk i+1 and the outputs of chunk i, so
    // its Q K^T issues while this group writes outputs.  Without it (one
    // chunk's Q/K in the ring, or one P buffer), chunk i at the top of its
    // iteration, once its slot has been reloaded.
    if (ROT && look) {
      for (int i = 0; i < 2 && i < nck && alive; ++i) alive = rotate_chunk(i);
    }
    if (look) {
      for (int i = -1; i < nck && alive; ++i) {
        if (i + 1 < nck && !ptilde(i + 1)) { alive = false; break; }
        if (ROT && i + 2 < nck && i >= 0 && !rotate_chunk(i + 2)) { alive = false; break; }
        if (i < 0) continue;
        if (fast) frame_advance(c, n, inv_g(i));
        if (!out_chunk(i, c)) { alive = false; break; }
      }
    } else {
      for (int i = 0; i < nck && alive; ++i) {
        if (ROT && !rotate_chunk(i)) { alive = false; break; }
        if (!ptilde(i)) { alive = false; break; }
        if (fast) frame_advance(c, n, inv_g(i));
        if (!out_chunk(i, c)) { alive = false; break; }
      }
    }
    if (eo == 0) bulk_wait_group0();
    }
  }

}

// Initialises the barriers of layout Cfg<C, DK, DVT, SO> (one thread).
template <int C, int DK, int DVT, bool SO>
__device__ __forceinline__ void init_barriers(uint32_t sbase) {
  using L = Cfg<C, DK, DVT, SO>;
  auto bar = [&](int i) { return sbase + L::oBar + 8 * i; };
  for (int i = 0; i < L::NQK; ++i) {
    mbar_init(bar(L::bQkFull + i), 1);
    mbar_init(bar(L::bQkEmpty + i), SO ? 1 : 2);  // main pass: both issuers read the slot
  }
  for (int i = 0; i < L::NV; ++i) {
    mbar_init(bar(L::bVFull + i), 1);
    mbar_init(bar(L::bVEmpty + i), 1);
    mbar_init(bar(L::bWReady + i), kGroup);
  }
  for (int i = 0; i < L::H; ++i) {
    mbar_init(bar(L::bSRead + i), kGroup);
    mbar_init(bar(L::bSFull + i), 1);
  }
  for (int i = 0; i < L::NSB; ++i) {
    mbar_init(bar(L::bSbReady + i), kGroup);
    mbar_init(bar(L::bSbFree + i), 1);
  }
  for (int i = 0; i < L::NP; ++i) {
    mbar_init(bar(L::bPFull + i), 1);
    mbar_init(bar(L::bPFree + i), 1);
    mbar_init(bar(L::bPtReady + i), kGroup);
  }
  for (int i = 0; i < L::NO; ++i) {
    mbar_init(bar(L::bOFull + i), 1);
    mbar_init(bar(L::bOFree + i), kGroup);
  }
  mbar_init(bar(L::bFin), SO ? 1 : 2);
  for (int i = 0; i < L::NV; ++i) mbar_init(bar(L::bSDone + i), 1);
  mbar_init(bar(L::bNever), 1);  // nothing ever arrives here (failure-path test)
  for (int i = 0; i < L::NQK; ++i) mbar_init(bar(L::bQkRot + i), kGroup);
}

// REV: time reversed (out_m sums over keys n >= m; see chunk_roles).
template <int C, int DK, int DVT, bool SO, bool NORM, bool ROT, bool REV>
__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmo,
                const TcParams p) {
  using L = Cfg<C, DK, DVT, SO>;
  extern __shared__ uint8_t smem_raw[];
  // Align by pointer arithmetic on the __shared__ array itself (not through an
  // integer), so the compiler keeps every access below in the shared window.
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(sm);
  float* pw = reinterpret_cast<float*>(sm + L::oPw);  // pw[d] = gamma^d, d = 0..C
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::oAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::oSlot);
  const int warp = threadIdx.x >> 5;
  float inv_gC = 1.f;

  // ---- set-up ----
  // The first chunks' slots are free, so for a split sequence (every CTA in
  // the first wave, the latency chain of pre-pass and main pass) the producer
  // thread issues their loads as soon as the barriers exist, before the wait
  // for gamma, the tables and the TMEM allocation.  Measured: mid -1.5 us,
  // long -1.5 us; with several waves of unsplit CTAs (7B-shaped) the early
  // burst cost 2%, so it is off there.
  const CtaPos pos = cta_pos<SO>(p);
  const float g = p.gamma[pos.bh % p.H];  // issued first: its latency overlaps the set-up
  const int c_begin = pos.seg * pos.seg_chunks;
  const int nck = min(c_begin + pos.seg_chunks, p.n_chunks) - c_begin;
  const int pre = pos.nseg > 1 ? max(0, min(nck, min(L::NV, L::NQK / L::H))) : 0;
  if (threadIdx.x == 0) {
    init_barriers<C, DK, DVT, SO>(sbase);
    *abort_flag = 0;
    fence_mbar_init();
    if (!SO) prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
    if (!SO) prefetch_tensormap(&tmo);
    for (int i = 0; i < pre; ++i) {
      const int j = SO ? c_begin + nck - 1 - i : c_begin + i;  // the roles' chunk order
      const int row = (REV ? p.n_chunks - 1 - j : j) * C;
      load_v<L, SO>(sbase, &tmv, i, row, pos.dvt * DVT, pos.bh);
      for (int hh = 0; hh < L::H; ++hh) load_qk<L, SO>(sbase, &tmq, &tmk, i * L::H + hh, hh, row, pos.bh);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  const float lg = g > 0.f ? log2f(g) : 0.f;
  const bool fast = g > 0.f && (float)C * lg >= kMinChunkDecayLog2;
  for (int d = threadIdx.x; d <= C; d += blockDim.x) pw[d] = gamma_pow(g, lg, (float)d);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (fast) inv_gC = 1.f / pw[C];
  // The main pass may start its CTAs now.  This comes after the TMEM
  // allocation, so a main-pass CTA that lands on this SM and waits for this
  // grid can never hold the columns this CTA still needs.
  if (SO) griddep_launch_dependents();

  const RoleCtx x{&tmq, &tmk, &tmv, &tmo, sm, tmem, inv_gC, pre};
  if (fast) chunk_roles<C, DK, DVT, SO, true, NORM, ROT, REV>(p, x);
  else chunk_roles<C, DK, DVT, SO, false, NORM, ROT, REV>(p, x);

  // ---- teardown: every MMA has completed, every load landed, every store read ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  write_final_state<C, DK, DVT, SO>(p, sm, tmem);
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

}  // namespace

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
bool make_map(CUtensorMap* m, const void* base, int d, int N, int BH, int rows, int ld) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  if (ld <= 0) ld = d;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)ld * 2 * (cuuint64_t)N};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// [B][N][H][dv] bf16 outputs (heads concatenated per token) viewed in 4-D as
// (channel, head, token, batch row), boxes of 64 channels x 1 head x `rows`
// tokens, 128-byte swizzle: one CTA's tile of one head.
bool make_map_heads(CUtensorMap* m, const void* base, int dv, int H, int N, int B, int rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)dv, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)dv * 2, (cuuint64_t)dv * 2 * H, (cuuint64_t)dv * 2 * H * (cuuint64_t)N};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int C, int DK, int DVT, bool SO, bool NORM, bool ROT, bool REV>
cudaError_t launch_one(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                       const CUtensorMap& mo, const TcParams& p, int grid, bool pdl, cudaStream_t s) {
  using L = Cfg<C, DK, DVT, SO>;
  auto kern = chunk_tc_kernel<C, DK, DVT, SO, NORM, ROT, REV>;
  // The shared-memory opt-in is a per-device function attribute: set it once per device.
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int C, int DK, int DVT, bool NORM, bool ROT, bool REV>
cudaError_t launch_pair(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const CUtensorMap& mo, const TcParams& p, cudaStream_t s) {
  const bool split = p.segments > 1;
  const int n_cut = p.BH * p.n_dv_tiles - p.full_units;
  if (split) {
    cudaError_t e = launch_one<C, DK, DVT, true, false, ROT, REV>(mq, mk, mv, mo, p, n_cut * (p.segments - 1), false, s);
    if (e != cudaSuccess) return e;
  }
  return launch_one<C, DK, DVT, false, NORM, ROT, REV>(mq, mk, mv, mo, p, p.full_units + n_cut * p.segments, split,
                                                       s);
}

// The variant for these tile sizes.
template <bool NORM, bool REV>
cudaError_t launch_variant_all(int chunk, int dkt, bool t128, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, const CUtensorMap& mo, const TcParams& p, cudaStream_t s);

// The variants for these tile sizes (with the fused rotation, or without it).
template <bool NORM, bool ROT>
cudaError_t launch_variant(int chunk, int dkt, bool t128, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const CUtensorMap& mo, const TcParams& p, cudaStream_t s) {
  if constexpr (ROT) {
    if (chunk == 64 && dkt == 128) return t128 ? launch_pair<64, 128, 128, NORM, ROT, false>(mq, mk, mv, mo, p, s)
                                               : launch_pair<64, 128, 64, NORM, ROT, false>(mq, mk, mv, mo, p, s);
    if (chunk == 64 && dkt == 256) return t128 ? launch_pair<64, 256, 128, NORM, ROT, false>(mq, mk, mv, mo, p, s)
                                               : launch_pair<64, 256, 64, NORM, ROT, false>(mq, mk, mv, mo, p, s);
    if (chunk == 128 && dkt == 128) return t128 ? launch_pair<128, 128, 128, NORM, ROT, false>(mq, mk, mv, mo, p, s)
                                                : launch_pair<128, 128, 64, NORM, ROT, false>(mq, mk, mv, mo, p, s);
    if (chunk == 128 && dkt == 256) return t128 ? launch_pair<128, 256, 128, NORM, ROT, false>(mq, mk, mv, mo, p, s)
                                                : launch_pair<128, 256, 64, NORM, ROT, false>(mq, mk, mv, mo, p, s);
    return cudaErrorNotSupported;
  } else {
    return launch_variant_all<NORM, false>(chunk, dkt, t128, mq, mk, mv, mo, p, s);
  }
}

template <bool NORM, bool REV>
cudaError_t launch_variant_all(int chunk, int dkt, bool t128, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, const CUtensorMap& mo, const TcParams& p, cudaStream_t s) {
  if (chunk == 64 && dkt == 128) return t128 ? launch_pair<64, 128, 128, NORM, false, REV>(mq, mk, mv, mo, p, s)
                                             : launch_pair<64, 128, 64, NORM, false, REV>(mq, mk, mv, mo, p, s);
  if (chunk == 128 && dkt == 128) return t128 ? launch_pair<128, 128, 128, NORM, false, REV>(mq, mk, mv, mo, p, s)
                                              : launch_pair<128, 128, 64, NORM, false, REV>(mq, mk, mv, mo, p, s);
  if (chunk == 64 && dkt == 256) return t128 ? launch_pair<64, 256, 128, NORM, false, REV>(mq, mk, mv, mo, p, s)
                                             : launch_pair<64, 256, 64, NORM, false, REV>(mq, mk, mv, mo, p, s);
  if (chunk == 128 && dkt == 256) return t128 ? launch_pair<128, 256, 128, NORM, false, REV>(mq, mk, mv, mo, p, s)
                                              : launch_pair<128, 256, 64, NORM, false, REV>(mq, mk, mv, mo, p, s);
  if constexpr (!NORM) {
    if (chunk == 64 && dkt == 512 && !t128) return launch_pair<64, 512, 64, false, false, REV>(mq, mk, mv, mo, p, s);
  }
  return cudaErrorNotSupported;
}

// The value-tile width used for these sizes.
int pick_dvt(int dv) { return dv % 128 == 0 ? 128 : 64; }

}  // namespace

std::atomic<unsigned int> g_test_stall_us{0};

int chunk_tc_launch_count(const ChunkPlan& plan) { return plan.launches; }

namespace {

// The split of a plan with tile height `tile`: segments, chunks per segment,
// cut units and their workspace (see chunk_tc_plan).
struct Split {
  int n_chunks, segs, seg_chunks;
  long long cut;
  size_t ws;
};
Split split_for(long long units, int N, int tile, int num_sms, int dk_tile, int dvt, size_t ws_limit) {
  Split r;
  r.n_chunks = (N + tile - 1) / tile;
  r.cut = units;
  int segs = 1;
  if (num_sms > 0 && units < num_sms) {
    segs = (int)(num_sms / units);
  } else if (num_sms > 0 && units % num_sms != 0) {
    r.cut = units % num_sms;
    segs = (int)(num_sms / r.cut);
  }
  segs = std::max(1, std::min(segs, r.n_chunks / 4));
  int seg_chunks = r.n_chunks > 0 ? (r.n_chunks + segs - 1) / segs : 1;
  if (r.n_chunks > 0) segs = (r.n_chunks + seg_chunks - 1) / seg_chunks;  // no empty segment
  // segment states cover the padded tile (dk_tile rows, dvt columns) of each cut unit
  r.ws = segs > 1 ? sizeof(float) * (size_t)r.cut * (segs - 1) * dk_tile * (size_t)dvt : 0;
  if (segs <= 1 || (r.cut < units && r.ws > ws_limit)) {
    segs = 1;
    seg_chunks = std::max(1, r.n_chunks);
    r.cut = units;
    r.ws = 0;
  }
  r.segs = segs;
  r.seg_chunks = std::max(1, seg_chunks);
  return r;
}

}  // namespace

bool chunk_tc_plan(int B, int H, int N, int dk, int dv, int chunk, int num_sms, ChunkPlan* plan,
                   size_t ws_limit, int tile) {
  // The chunk length is a tiling choice that leaves the result unchanged
  // (every chunk length computes the same sums, up to rounding order), so the
  // kernels run 128-token tiles (full-height tensor-core tiles, half as many
  // per-chunk steps as 64-token ones: mid -10%, its gradients -9%), unless
  // 64-token tiles give more CTAs (a short sequence with few units, where the
  // segments are capped at n_chunks / 4) or the caller fixes the tile.
  if (!(chunk == 32 || chunk == 64 || chunk == 128)) return false;
  if (!(tile == 0 || tile == 64 || tile == 128)) return false;
  if (dk < 16 || dk > 512 || dk % 16 != 0) return false;
  if (dv < 16 || dv > 1024 || dv % 16 != 0) return false;
  if (N < 0) return false;
  // above 256 query/key columns: 512-wide tiles with 64-token, 64-wide value tiles
  const bool wide = dk > 256;
  if (wide && tile == 128) return false;
  if (wide) tile = 64;
  const int dvt = wide ? 64 : pick_dvt(dv);
  plan->dk_tile = dk <= 128 ? 128 : dk <= 256 ? 256 : 512;
  plan->dvt = dvt;
  plan->n_dv_tiles = (dv + dvt - 1) / dvt;
  const long long units = (long long)B * H * plan->n_dv_tiles;
  if (units > (1LL << 30)) return false;
  // Enough segments that every SM gets a CTA, each segment at least 4 chunks:
  // with fewer units than SMs every unit is cut; with more, the units of the
  // last, partial wave are cut so that it holds about as many CTAs as there
  // are SMs (the other units run whole), if their segment states fit within
  // ws_limit bytes.
  Split sp = split_for(units, N, tile ? tile : 128, num_sms, plan->dk_tile, dvt, ws_limit);
  plan->chunk = tile ? tile : 128;
  if (tile == 0) {
    const Split s64 = split_for(units, N, 64, num_sms, plan->dk_tile, dvt, ws_limit);
    auto ctas = [&](const Split& x) { return units - x.cut + x.cut * x.segs; };
    if (ctas(s64) > ctas(sp)) {
      sp = s64;
      plan->chunk = 64;
    }
  }
  plan->n_chunks = sp.n_chunks;
  plan->segments = sp.segs;
  plan->seg_chunks = sp.seg_chunks;
  plan->full_units = sp.segs > 1 ? (int)(units - sp.cut) : (int)units;
  plan->workspace_bytes = sp.ws;
  plan->launches = sp.segs > 1 ? 2 : 1;
  if (plan->full_units + sp.cut * sp.segs > INT32_MAX) return false;
  return true;
}

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* gamma,
                            const float* state_in, void* out, float* state_out, int B, int H, int N,
                            int dk, int dv, const ChunkPlan& plan, float* workspace,
                            const ChunkNorm* norm, float scale, cudaStream_t s, const ChunkRotation* rot,
                            bool rev, int ldqk) {
  const int BH = B * H;
  const int chunk = plan.chunk;
  if (rev && (norm || rot)) return cudaErrorNotSupported;
  // GroupNorm statistics need a head's whole row, unpadded, in one CTA
  if (norm && (plan.n_dv_tiles != 1 || plan.dvt != dv)) return cudaErrorNotSupported;
  if (norm && rot) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, q, dk, N, BH, chunk, ldqk) || !make_map(&mk, k, dk, N, BH, chunk, ldqk) ||
      !make_map(&mv, v, dv, N, BH, chunk) ||
      !(norm ? make_map_heads(&mo, out, dv, H, N, B, chunk) : make_map(&mo, out, dv, N, BH, chunk)))
    return cudaErrorInvalidValue;
  TcParams p;
  p.gamma = gamma;
  p.state_in = state_in;
  p.state_out = state_out;
  p.ws = workspace;
  p.norm_w = norm ? norm->weight : nullptr;
  p.norm_b = norm ? norm->bias : nullptr;
  p.norm_eps = norm ? norm->eps : 0.f;
  p.H = H;
  p.N = N;
  p.dv = dv;
  p.dk = dk;
  p.n_dv_tiles = plan.n_dv_tiles;
  p.BH = BH;
  p.segments = plan.segments;
  p.seg_chunks = plan.seg_chunks;
  p.n_chunks = plan.n_chunks;
  p.full_units = plan.full_units;
  p.scale = scale > 0.f ? scale : (float)(1.0 / std::sqrt((double)dk));
  p.test_stall_us = g_test_stall_us.load(std::memory_order_relaxed);
  p.theta = rot ? rot->theta : nullptr;
  p.n0 = rot ? rot->n0 : 0;
  const bool t128 = plan.dvt == 128;
  const int dkt = plan.dk_tile;
  if (rev) return launch_variant_all<false, true>(chunk, dkt, t128, mq, mk, mv, mo, p, s);
  if (norm) return launch_variant<true, false>(chunk, dkt, t128, mq, mk, mv, mo, p, s);
  if (rot) return launch_variant<false, true>(chunk, dkt, t128, mq, mk, mv, mo, p, s);
  return launch_variant<false, false>(chunk, dkt, t128, mq, mk, mv, mo, p, s);
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
