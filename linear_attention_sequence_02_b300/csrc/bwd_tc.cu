// bwd_tc.cu -- gradients of retention on the tensor cores, each computed as a
// retention forward of permuted operands by the chunkwise kernel (chunk_tc.cu).
//
// The gradients of the forward started from S0, for the loss
// <dout, out> + <dS, S_N> (s = 1/sqrt(dk), g = gamma_h), are
//
//   dq_n  = s [ sum_{m<=n} g^(n-m) (dout_n . v_m) k_m + g^(n+1) dout_n S0^T ]
//   dk_m  = s sum_{n>=m} g^(n-m) (v_m . dout_n) q_n + g^(N-1-m) v_m dS^T
//   dv_m  = s sum_{n>=m} g^(n-m) (k_m . q_n) dout_n + g^(N-1-m) k_m dS
//   dS0   = s sum_n g^(n+1) q_n^T dout_n + g^N dS
//
// The first line is the forward of "3. The Chunkwise Recurrent Representation
// ..." ("RetNet Guide: Retentive Networks & The Impossible Triangle") with
// query dout, key v, value k and starting state S0^T, at query factor s.  With
// time reversed (t = N-1-m), the second and third are the same forward of
// (v, dout, q) and (k, q, dout) started from X = dS^T / (s g) and dS / (s g):
// the forward's starting-state term s g^(t+1) v_t X is g^t v_t dS^T.  dS0 is
// s g times the final state of the reversed (k, q, dout) forward.  A head
// with g = 0 has no such X: it runs from a zero state and its final-state
// term, which reaches only the last token (0^0 = 1), is added afterwards (so
// does a head with g <= 2^-64, where 1/(s g) could overflow and every other
// power of g is negligible).
//
// So one call is: a gather kernel that stacks the permuted (and, for the
// reversed problems, row-reversed) operands into batch-stacked tensors; a
// kernel that prepares the starting states; one chunkwise forward per
// operand shape (one when dk == dv, the three problems stacked on the batch
// axis; two otherwise); and the same gather kernel run backwards to place the
// results, then dS0 and the decay-0 term.  Scratch is allocated
// stream-ordered on the caller's stream.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "internal.h"

namespace ret {
namespace {

constexpr int kMaxJobs = 9;
// Decays at or below this are treated as 0 by the starting states: 1/(s g)
// could overflow, and every power g^t with t >= 1 is below 2^-64 there, so
// only the t = 0 term (added by zero_decay_term_kernel) is kept.
constexpr float kTinyDecay = 5.42101086e-20f;  // 2^-64

// Copy of a [BH][N][w] bf16 tensor into another, rows optionally reversed in
// each head (row n of dst is row N-1-n of src).
struct SeqJob {
  const uint4* src;
  uint4* dst;
  int w16;      // row width in 16-byte units
  int reverse;
};
struct SeqJobs {
  SeqJob job[kMaxJobs];
  int BH, N;
};

// grid: (row blocks of one head, head, job).  A block copies kRowIters
// groups of `rows` = 256 / w16 rows; thread t moves 16-byte unit t % w16 of
// row t / w16 of each group, so every row is one contiguous run of a warp's
// stores and every load is a whole row of the source.
constexpr int kRowIters = 4;
__global__ void __launch_bounds__(256) seq_gather_kernel(const __grid_constant__ SeqJobs J) {
  const SeqJob j = J.job[blockIdx.z];
  const int w16 = j.w16;
  const int rows = 256 / w16;  // rows per group
  const int t = threadIdx.x;
  const int r = t / w16, c = t - r * w16;
  if (r >= rows) return;
  const size_t head = (size_t)blockIdx.y * J.N;
  const int n0 = blockIdx.x * rows * kRowIters + r;
  uint4 x[kRowIters];
#pragma unroll
  for (int it = 0; it < kRowIters; ++it) {
    const int n = n0 + it * rows;
    if (n < J.N) {
      const int sn = j.reverse ? J.N - 1 - n : n;
      x[it] = __ldcs(j.src + (head + sn) * w16 + c);
    }
  }
#pragma unroll
  for (int it = 0; it < kRowIters; ++it) {
    const int n = n0 + it * rows;
    if (n < J.N) __stcs(j.dst + (head + n) * w16 + c, x[it]);
  }
}

// Starting states and dS0: dst = f(h) * src or f(h) * src^T per head, src
// [BH][r][c] float32 (NULL: zero), dst [BH][c][r] when transposed; f is 1,
// 1/(s g) (0 where g = 0) or s g.
enum StateScale { kOne = 0, kInvSG = 1, kSG = 2 };
struct StateJob {
  const float* src;
  float* dst;
  int transpose;
  int scale;
};
struct StateJobs {
  StateJob job[3];
  const float* gamma;
  int H, r, c;  // source rows, columns
  float s;
};

// grid: (32x32 tiles of one head, BH, job); block 32 x 8.
__global__ void __launch_bounds__(256) state_prep_kernel(const __grid_constant__ StateJobs J) {
  __shared__ float tile[32][33];
  const StateJob j = J.job[blockIdx.z];
  const int bh = blockIdx.y;
  const int tiles_c = (J.c + 31) / 32;
  const int r0 = (blockIdx.x / tiles_c) * 32, c0 = (blockIdx.x % tiles_c) * 32;
  const float g = J.gamma[bh % J.H];
  float f = 1.f;
  if (j.scale == kInvSG) f = g > kTinyDecay ? 1.f / (J.s * g) : 0.f;
  if (j.scale == kSG) f = J.s * g;
  const size_t head = (size_t)bh * J.r * J.c;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int y = ty; y < 32; y += 8) {
    const int r = r0 + y, c = c0 + tx;
    float x = 0.f;
    if (j.src && r < J.r && c < J.c) x = f * j.src[head + (size_t)r * J.c + c];
    if (!j.transpose) {
      if (r < J.r && c < J.c) j.dst[head + (size_t)r * J.c + c] = x;
    } else {
      tile[y][tx] = x;
    }
  }
  if (!j.transpose) return;
  __syncthreads();
  // dst is [c][r]: row c0 + y, column r0 + tx
  for (int y = ty; y < 32; y += 8) {
    const int c = c0 + y, r = r0 + tx;
    if (r < J.r && c < J.c) j.dst[head + (size_t)c * J.r + r] = tile[tx][y];
  }
}

// Decay-0 heads (g <= kTinyDecay) with a final-state gradient:
// dk_{N-1} += v_{N-1} dS^T and dv_{N-1} += k_{N-1} dS (the only terms of
// g^(N-1-m) dS that survive).  One block per head; other heads return at once.
__global__ void __launch_bounds__(256) zero_decay_term_kernel(const __nv_bfloat16* k, const __nv_bfloat16* v,
                                                              const float* dS, const float* gamma,
                                                              __nv_bfloat16* dk_out, __nv_bfloat16* dv_out, int H,
                                                              int N, int dk, int dv) {
  const int bh = blockIdx.x;
  if (gamma[bh % H] > kTinyDecay) return;
  const size_t last = (size_t)bh * N + (N - 1);
  const float* S = dS + (size_t)bh * dk * dv;
  for (int i = threadIdx.x; i < dk; i += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < dv; ++j) acc = fmaf(__bfloat162float(v[last * dv + j]), S[(size_t)i * dv + j], acc);
    __nv_bfloat16* o = dk_out + last * dk + i;
    *o = __float2bfloat16_rn(__bfloat162float(*o) + acc);
  }
  for (int j = threadIdx.x; j < dv; j += blockDim.x) {
    float acc = 0.f;
    for (int i = 0; i < dk; ++i) acc = fmaf(__bfloat162float(k[last * dk + i]), S[(size_t)i * dv + j], acc);
    __nv_bfloat16* o = dv_out + last * dv + j;
    *o = __float2bfloat16_rn(__bfloat162float(*o) + acc);
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int num_sms_current() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

cudaError_t launch_seq(const SeqJobs& J, int n_jobs, cudaStream_t s) {
  if (n_jobs == 0) return cudaSuccess;
  int min_rows = 256;
  for (int i = 0; i < n_jobs; ++i) min_rows = std::min(min_rows, 256 / J.job[i].w16);
  const int blocks = (J.N + min_rows * kRowIters - 1) / (min_rows * kRowIters);
  seq_gather_kernel<<<dim3(blocks, J.BH, n_jobs), 256, 0, s>>>(J);
  return cudaGetLastError();
}

// One chunkwise forward over the batch-stacked problems of one operand shape.
struct Group {
  int parts;       // problems stacked on the batch axis
  int dkp, dvp;    // the forward's query/key and value widths
  ChunkPlan plan;
  __nv_bfloat16 *q, *k, *v, *o;  // [parts*B][H][N][dkp or dvp]
  float* state_in;               // [parts*B][H][dkp][dvp] or NULL
  float* state_out;              // likewise, or NULL
  float* ws;                     // segment scratch of the forward
};

}  // namespace

bool backward_tc_supported(int dk, int dv) {
  return dk % 16 == 0 && dv % 16 == 0 && dk >= 16 && dv >= 16 && dk <= 256 && dv <= 256;
}

cudaError_t launch_backward_tc(const void* q, const void* k, const void* v, const float* gamma, const float* state_in,
                               const void* dout, const float* dstate, void* dq, void* dk_out, void* dv_out,
                               float* dstate_in, int B, int H, int N, int dk, int dv, cudaStream_t s) {
  const int sms = num_sms_current();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int BH = B * H;
  if (BH > 65535) return cudaErrorNotSupported;  // heads on the gather grid's y axis
  const float scale = (float)(1.0 / std::sqrt((double)dk));
  const int chunk = N >= 4096 ? 128 : 64;
  const bool same = dk == dv;
  // Problems: 0 = dq (dout, v, k | S0^T), 1 = dk (rev v, rev dout, rev q | dS^T/(s g)),
  // 2 = dv (rev k, rev q, rev dout | dS/(s g)).  Problems 0 and 1 have the
  // shape (dv, dk), problem 2 (dk, dv).
  Group grp[2];
  const int n_groups = same ? 1 : 2;
  grp[0].parts = same ? 3 : 2;
  grp[0].dkp = dv;
  grp[0].dvp = dk;
  if (!same) {
    grp[1].parts = 1;
    grp[1].dkp = dk;
    grp[1].dvp = dv;
  }
  const bool any_state = state_in != nullptr || dstate != nullptr;
  size_t bytes = 0;
  size_t off[2][7];
  for (int gi = 0; gi < n_groups; ++gi) {
    Group& G = grp[gi];
    if (!chunk_tc_plan(G.parts * B, H, N, G.dkp, G.dvp, chunk, sms, &G.plan)) return cudaErrorNotSupported;
    const size_t rows = (size_t)G.parts * BH * N, st = sizeof(float) * (size_t)G.parts * BH * G.dkp * G.dvp;
    const size_t sz[7] = {rows * G.dkp * 2, rows * G.dkp * 2, rows * G.dvp * 2, rows * G.dvp * 2,
                          any_state ? st : 0, dstate_in ? st : 0, G.plan.workspace_bytes};
    for (int i = 0; i < 7; ++i) {
      off[gi][i] = bytes;
      bytes += align256(sz[i]);
    }
  }
  char* base = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&base), bytes, s);
  if (e != cudaSuccess) return e;
  for (int gi = 0; gi < n_groups; ++gi) {
    Group& G = grp[gi];
    G.q = reinterpret_cast<__nv_bfloat16*>(base + off[gi][0]);
    G.k = reinterpret_cast<__nv_bfloat16*>(base + off[gi][1]);
    G.v = reinterpret_cast<__nv_bfloat16*>(base + off[gi][2]);
    G.o = reinterpret_cast<__nv_bfloat16*>(base + off[gi][3]);
    G.state_in = any_state ? reinterpret_cast<float*>(base + off[gi][4]) : nullptr;
    G.state_out = dstate_in ? reinterpret_cast<float*>(base + off[gi][5]) : nullptr;
    G.ws = G.plan.workspace_bytes ? reinterpret_cast<float*>(base + off[gi][6]) : nullptr;
  }
  // where problem p lives: its group and its part inside the group
  const int pg[3] = {0, 0, same ? 0 : 1}, pp[3] = {0, 1, same ? 2 : 0};
  auto part_ptr = [&](__nv_bfloat16* t, int p, int width) {
    return reinterpret_cast<uint4*>(t + (size_t)pp[p] * BH * N * width);
  };
  const uint4 *Q = static_cast<const uint4*>(q), *K = static_cast<const uint4*>(k), *V = static_cast<const uint4*>(v),
              *DO = static_cast<const uint4*>(dout);
  const int qk16 = dk / 8, v16 = dv / 8;

  // 1. operands: (query, key, value) of each problem
  SeqJobs in{};
  in.BH = BH;
  in.N = N;
  int nj = 0;
  auto add = [&](SeqJobs& J, const uint4* src, uint4* dst, int w16, int rev) { J.job[nj++] = SeqJob{src, dst, w16, rev}; };
  {
    Group &G0 = grp[pg[0]], &G1 = grp[pg[1]], &G2 = grp[pg[2]];
    add(in, DO, part_ptr(G0.q, 0, G0.dkp), v16, 0);
    add(in, V, part_ptr(G0.k, 0, G0.dkp), v16, 0);
    add(in, K, part_ptr(G0.v, 0, G0.dvp), qk16, 0);
    add(in, V, part_ptr(G1.q, 1, G1.dkp), v16, 1);
    add(in, DO, part_ptr(G1.k, 1, G1.dkp), v16, 1);
    add(in, Q, part_ptr(G1.v, 1, G1.dvp), qk16, 1);
    add(in, K, part_ptr(G2.q, 2, G2.dkp), qk16, 1);
    add(in, Q, part_ptr(G2.k, 2, G2.dkp), qk16, 1);
    add(in, DO, part_ptr(G2.v, 2, G2.dvp), v16, 1);
  }
  e = launch_seq(in, nj, s);

  // 2. starting states
  if (e == cudaSuccess && any_state) {
    for (int gi = 0; gi < n_groups && e == cudaSuccess; ++gi) {
      Group& G = grp[gi];
      StateJobs J{};
      J.gamma = gamma;
      J.H = H;
      J.r = dk;
      J.c = dv;
      J.s = scale;
      int n = 0;
      for (int p = 0; p < 3; ++p) {
        if (pg[p] != gi) continue;
        float* dst = G.state_in + (size_t)pp[p] * BH * dk * dv;
        if (p == 0) J.job[n++] = StateJob{state_in, dst, 1, kOne};
        if (p == 1) J.job[n++] = StateJob{dstate, dst, 1, kInvSG};
        if (p == 2) J.job[n++] = StateJob{dstate, dst, 0, kInvSG};
      }
      const int tiles = ((dk + 31) / 32) * ((dv + 31) / 32);
      state_prep_kernel<<<dim3(tiles, BH, n), dim3(32, 8), 0, s>>>(J);
      e = cudaGetLastError();
    }
  }

  // 3. the forwards
  for (int gi = 0; gi < n_groups && e == cudaSuccess; ++gi) {
    Group& G = grp[gi];
    e = launch_chunk_tc(G.q, G.k, G.v, gamma, G.state_in, G.o, G.state_out, G.parts * B, H, N, G.dkp, G.dvp, G.plan,
                        G.ws, nullptr, scale, s);
  }

  // 4. results into place: dq as is, dk and dv with their rows reversed back
  if (e == cudaSuccess) {
    SeqJobs out{};
    out.BH = BH;
    out.N = N;
    nj = 0;
    add(out, part_ptr(grp[pg[0]].o, 0, grp[pg[0]].dvp), static_cast<uint4*>(dq), qk16, 0);
    add(out, part_ptr(grp[pg[1]].o, 1, grp[pg[1]].dvp), static_cast<uint4*>(dk_out), qk16, 1);
    add(out, part_ptr(grp[pg[2]].o, 2, grp[pg[2]].dvp), static_cast<uint4*>(dv_out), v16, 1);
    e = launch_seq(out, nj, s);
  }
  // 5. dS0 = s g times the final state of the dv problem
  if (e == cudaSuccess && dstate_in) {
    StateJobs J{};
    J.gamma = gamma;
    J.H = H;
    J.r = dk;
    J.c = dv;
    J.s = scale;
    J.job[0] = StateJob{grp[pg[2]].state_out + (size_t)pp[2] * BH * dk * dv, dstate_in, 0, kSG};
    const int tiles = ((dk + 31) / 32) * ((dv + 31) / 32);
    state_prep_kernel<<<dim3(tiles, BH, 1), dim3(32, 8), 0, s>>>(J);
    e = cudaGetLastError();
  }
  // 6. decay-0 heads: the final-state gradient's last-token term
  if (e == cudaSuccess && dstate) {
    zero_decay_term_kernel<<<BH, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(k),
                                              static_cast<const __nv_bfloat16*>(v), dstate, gamma,
                                              static_cast<__nv_bfloat16*>(dk_out),
                                              static_cast<__nv_bfloat16*>(dv_out), H, N, dk, dv);
    e = cudaGetLastError();
  }
  const cudaError_t e2 = cudaFreeAsync(base, s);
  return e != cudaSuccess ? e : e2;
}

int backward_tc_launches(int B, int H, int N, int dk, int dv, bool has_state_in, bool has_dstate, bool want_dstate_in) {
  const int sms = 148;
  const int chunk = N >= 4096 ? 128 : 64;
  int n = 2;  // gather in, gather out
  if (has_state_in || has_dstate) n += dk == dv ? 1 : 2;
  if (want_dstate_in) n += 1;
  if (has_dstate) n += 1;
  const int groups = dk == dv ? 1 : 2;
  for (int gi = 0; gi < groups; ++gi) {
    ChunkPlan plan;
    const int parts = dk == dv ? 3 : (gi == 0 ? 2 : 1);
    if (!chunk_tc_plan(parts * B, H, N, gi == 0 ? dv : dk, gi == 0 ? dk : dv, chunk, sms, &plan)) return -1;
    n += chunk_tc_launch_count(plan);
  }
  return n;
}

}  // namespace ret
