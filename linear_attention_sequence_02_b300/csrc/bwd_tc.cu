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
// So one call is: a kernel that prepares the starting states, the three
// forwards read straight from the caller's tensors and written straight into
// the gradients (the chunkwise kernel's time-reversed mode takes the rows of
// the second and third from the last to the first), then dS0 and the decay-0
// term.  The three forwards are independent; they run on three streams (the
// caller's and two of the library's own, forked and joined with events), each
// planned for a third of the SMs, so together they fill the GPU like one
// launch.  Scratch is allocated stream-ordered on the caller's stream.
//
// A forward is linear in a split of its query/key width: with q = [q1 q2] and
// k = [k1 k2], (q_n . k_m) = (q1_n . k1_m) + (q2_n . k2_m) and the state's
// rows split the same way, so the forward of (q, k, v) from S is the sum of
// the forwards of (q1, k1, v) from S's first rows and (q2, k2, v) from the
// rest.  Forwards whose query/key width is above 256 (dq's and dk's when
// dv > 256) run as 256-column parts on the 128-token tiles (q and k read in
// place with the row stride of the full width; each part's rows of the
// starting and final states copied to and from packed buffers), the first
// part into the gradient, the others into scratch, then summed into it.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace ret {
namespace {

// Decays at or below this are treated as 0 by the starting states: 1/(s g)
// could overflow, and every power g^t with t >= 1 is below 2^-64 there, so
// only the t = 0 term (added by zero_decay_term_kernel) is kept.
constexpr float kTinyDecay = 5.42101086e-20f;  // 2^-64

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

// Two streams of the library's own per device, created on the first call
// (make that call outside stream capture), and the events that fork the
// gradient call's work onto them and join it back.  The lock is held while a
// call enqueues, so the events are never re-recorded before the waits on
// them are enqueued.
constexpr int kMaxDevices = 64;
struct Aux {
  cudaStream_t st[2];
  cudaEvent_t fork, join[2];
  bool ready;
};
std::mutex g_aux_lock[kMaxDevices];
Aux g_aux[kMaxDevices];

cudaError_t aux_for(int dev, Aux** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  Aux& a = g_aux[dev];
  if (!a.ready) {
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&a.st[i], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&a.join[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    a.ready = true;
  }
  *out = &a;
  return cudaSuccess;
}

// The three forwards: 0 = dq (dout, v, k | S0^T), 1 = dk (v, dout, q |
// dS^T/(s g), time reversed), 2 = dv (k, q, dout | dS/(s g), time reversed).
constexpr int kPartWidth = 256;  // query/key columns of one part of a wide forward
constexpr int kMaxParts = 2;     // widths up to 512
struct Problem {
  const void *q, *k, *v;
  void* o;
  int dkp, dvp;     // the forward's query/key and value widths
  bool rev;
  int parts;        // ceil(dkp / kPartWidth)
  ChunkPlan plan[kMaxParts];
  float* state_in;  // or NULL (zero)
  float* state_out; // or NULL
  float* ws[kMaxParts];
  __nv_bfloat16* partial[kMaxParts];  // outputs of parts 1.. (part 0 writes o)
  float* part_in[kMaxParts];   // with several parts: each part's rows of the states, packed per head
  float* part_out[kMaxParts];
};

// dst += src, bf16, n elements (a multiple of 8, both 16-byte aligned).
__global__ void __launch_bounds__(256) add_bf16_kernel(__nv_bfloat16* dst, const __nv_bfloat16* src, size_t n8) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    uint4 a = reinterpret_cast<uint4*>(dst)[i];
    const uint4 b = reinterpret_cast<const uint4*>(src)[i];
    uint32_t* pa = reinterpret_cast<uint32_t*>(&a);
    const uint32_t* pb = reinterpret_cast<const uint32_t*>(&b);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pa[e]));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pb[e]));
      const __nv_bfloat162 z = __floats2bfloat162_rn(x.x + y.x, x.y + y.y);
      pa[e] = *reinterpret_cast<const uint32_t*>(&z);
    }
    reinterpret_cast<uint4*>(dst)[i] = a;
  }
}

int backward_chunk(int N) { return N >= 4096 ? 128 : 64; }

}  // namespace

bool backward_tc_supported(int dk, int dv) {
  return dk % 16 == 0 && dv % 16 == 0 && dk >= 16 && dv >= 16 && dk <= 512 && dv <= 512;
}

cudaError_t launch_backward_tc(const void* q, const void* k, const void* v, const float* gamma, const float* state_in,
                               const void* dout, const float* dstate, void* dq, void* dk_out, void* dv_out,
                               float* dstate_in, int B, int H, int N, int dk, int dv, cudaStream_t s) {
  const int sms = num_sms_current();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int BH = B * H;
  if (BH > 65535) return cudaErrorNotSupported;  // heads on the state kernels' grid y axis
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const float scale = (float)(1.0 / std::sqrt((double)dk));
  const int chunk = backward_chunk(N);
  const int share = std::max(1, sms / 3);
  Problem P[3] = {};
  const void* ops[3][4] = {{dout, v, k, dq}, {v, dout, q, dk_out}, {k, q, dout, dv_out}};
  const int widths[3][2] = {{dv, dk}, {dv, dk}, {dk, dv}};
  for (int i = 0; i < 3; ++i) {
    P[i].q = ops[i][0];
    P[i].k = ops[i][1];
    P[i].v = ops[i][2];
    P[i].o = const_cast<void*>(ops[i][3]);
    P[i].dkp = widths[i][0];
    P[i].dvp = widths[i][1];
    P[i].rev = i > 0;
    P[i].parts = (P[i].dkp + kPartWidth - 1) / kPartWidth;
    if (P[i].parts > kMaxParts) return cudaErrorNotSupported;
  }
  const bool want_state[3] = {state_in != nullptr, dstate != nullptr, dstate != nullptr};
  const size_t st_bytes = sizeof(float) * (size_t)BH * dk * dv;
  size_t bytes = 0, off_in[3], off_ws[3][kMaxParts], off_part[3][kMaxParts], off_out = 0;
  for (int i = 0; i < 3; ++i) {
    off_in[i] = bytes;
    bytes += want_state[i] ? align256(st_bytes) : 0;
    for (int j = 0; j < P[i].parts; ++j) {
      const int w = std::min(kPartWidth, P[i].dkp - j * kPartWidth);
      if (!chunk_tc_plan(B, H, N, w, P[i].dvp, chunk, share, &P[i].plan[j])) return cudaErrorNotSupported;
      off_ws[i][j] = bytes;
      bytes += align256(P[i].plan[j].workspace_bytes);
      off_part[i][j] = bytes;
      bytes += j > 0 ? align256((size_t)BH * N * P[i].dvp * 2) : 0;
    }
  }
  // packed per-part state rows (only for problems in several parts)
  size_t off_pin[3][kMaxParts] = {}, off_pout[3][kMaxParts] = {};
  for (int i = 0; i < 3; ++i) {
    if (P[i].parts < 2) continue;
    for (int j = 0; j < P[i].parts; ++j) {
      const size_t w = (size_t)std::min(kPartWidth, P[i].dkp - j * kPartWidth);
      const size_t pb = sizeof(float) * (size_t)BH * w * P[i].dvp;
      off_pin[i][j] = bytes;
      bytes += want_state[i] ? align256(pb) : 0;
      off_pout[i][j] = bytes;
      bytes += (i == 2 && dstate_in) ? align256(pb) : 0;
    }
  }
  if (dstate_in) {
    off_out = bytes;
    bytes += align256(st_bytes);
  }
  char* base = nullptr;
  if (bytes > 0) {
    e = cudaMallocAsync(reinterpret_cast<void**>(&base), bytes, s);
    if (e != cudaSuccess) return e;
  }
  for (int i = 0; i < 3; ++i) {
    P[i].state_in = want_state[i] ? reinterpret_cast<float*>(base + off_in[i]) : nullptr;
    for (int j = 0; j < P[i].parts; ++j) {
      P[i].ws[j] = P[i].plan[j].workspace_bytes ? reinterpret_cast<float*>(base + off_ws[i][j]) : nullptr;
      P[i].partial[j] = j > 0 ? reinterpret_cast<__nv_bfloat16*>(base + off_part[i][j]) : nullptr;
      const bool multi = P[i].parts > 1;
      P[i].part_in[j] = multi && want_state[i] ? reinterpret_cast<float*>(base + off_pin[i][j]) : nullptr;
      P[i].part_out[j] = multi && i == 2 && dstate_in ? reinterpret_cast<float*>(base + off_pout[i][j]) : nullptr;
    }
  }
  if (dstate_in) P[2].state_out = reinterpret_cast<float*>(base + off_out);

  // 1. starting states: S0^T, dS^T/(s g), dS/(s g)
  const int tiles = ((dk + 31) / 32) * ((dv + 31) / 32);
  {
    StateJobs J{};
    J.gamma = gamma;
    J.H = H;
    J.r = dk;
    J.c = dv;
    J.s = scale;
    int n = 0;
    if (want_state[0]) J.job[n++] = StateJob{state_in, P[0].state_in, 1, kOne};
    if (want_state[1]) J.job[n++] = StateJob{dstate, P[1].state_in, 1, kInvSG};
    if (want_state[2]) J.job[n++] = StateJob{dstate, P[2].state_in, 0, kInvSG};
    if (n > 0) {
      state_prep_kernel<<<dim3(tiles, BH, n), dim3(32, 8), 0, s>>>(J);
      e = cudaGetLastError();
    }
  }

  // 2. the three forwards, forked onto three streams and joined back
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> hold(g_aux_lock[dev]);
    Aux* a = nullptr;
    e = aux_for(dev, &a);
    if (e == cudaSuccess) e = cudaEventRecord(a->fork, s);
    bool forked[2] = {false, false};
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
      e = cudaStreamWaitEvent(a->st[i], a->fork, 0);
      forked[i] = e == cudaSuccess;
    }
    const cudaStream_t where[3] = {s, forked[0] ? a->st[0] : s, forked[1] ? a->st[1] : s};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) {
      const Problem& X = P[i];
      // part j: query/key columns [256 j, 256 j + w) and the same rows of the states
      for (int j = 0; j < X.parts && e == cudaSuccess; ++j) {
        const int c0 = j * kPartWidth, w = std::min(kPartWidth, X.dkp - c0);
        // a part's rows of a head's state: w rows of dvp floats at row c0 of the dkp-row state
        const size_t head = sizeof(float) * (size_t)X.dkp * X.dvp, rows = sizeof(float) * (size_t)w * X.dvp;
        const size_t first = sizeof(float) * (size_t)c0 * X.dvp;
        const float* sin = X.state_in;
        float* sout = X.state_out;
        if (X.parts > 1) {
          if (X.state_in) {
            e = cudaMemcpy2DAsync(X.part_in[j], rows, reinterpret_cast<const char*>(X.state_in) + first, head, rows,
                                  BH, cudaMemcpyDeviceToDevice, where[i]);
            sin = X.part_in[j];
          }
          sout = X.part_out[j];
        }
        if (e == cudaSuccess)
          e = launch_chunk_tc(static_cast<const __nv_bfloat16*>(X.q) + c0, static_cast<const __nv_bfloat16*>(X.k) + c0,
                              X.v, gamma, sin, j == 0 ? X.o : X.partial[j], sout, B, H, N, w, X.dvp, X.plan[j],
                              X.ws[j], nullptr, scale, where[i], nullptr, X.rev, X.dkp);
        if (e == cudaSuccess && X.parts > 1 && X.state_out)
          e = cudaMemcpy2DAsync(reinterpret_cast<char*>(X.state_out) + first, head, X.part_out[j], rows, rows, BH,
                                cudaMemcpyDeviceToDevice, where[i]);
      }
      for (int j = 1; j < X.parts && e == cudaSuccess; ++j) {
        const size_t n8 = (size_t)BH * N * X.dvp / 8;
        const int blocks = (int)std::min<size_t>((n8 + 255) / 256, (size_t)sms * 8);
        add_bf16_kernel<<<blocks, 256, 0, where[i]>>>(static_cast<__nv_bfloat16*>(X.o), X.partial[j], n8);
        e = cudaGetLastError();
      }
    }
    // join whatever was forked, whether or not every launch went in
    for (int i = 0; i < 2; ++i) {
      if (!forked[i]) continue;
      cudaError_t ej = cudaEventRecord(a->join[i], a->st[i]);
      if (ej == cudaSuccess) ej = cudaStreamWaitEvent(s, a->join[i], 0);
      if (e == cudaSuccess) e = ej;
    }
  }
  // 3. dS0 = s g times the final state of the dv problem
  if (e == cudaSuccess && dstate_in) {
    StateJobs J{};
    J.gamma = gamma;
    J.H = H;
    J.r = dk;
    J.c = dv;
    J.s = scale;
    J.job[0] = StateJob{P[2].state_out, dstate_in, 0, kSG};
    state_prep_kernel<<<dim3(tiles, BH, 1), dim3(32, 8), 0, s>>>(J);
    e = cudaGetLastError();
  }
  // 4. decay-0 heads: the final-state gradient's last-token term
  if (e == cudaSuccess && dstate) {
    zero_decay_term_kernel<<<BH, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(k),
                                              static_cast<const __nv_bfloat16*>(v), dstate, gamma,
                                              static_cast<__nv_bfloat16*>(dk_out),
                                              static_cast<__nv_bfloat16*>(dv_out), H, N, dk, dv);
    e = cudaGetLastError();
  }
  if (base) {
    const cudaError_t e2 = cudaFreeAsync(base, s);
    if (e == cudaSuccess) e = e2;
  }
  return e;
}

int backward_tc_launches(int B, int H, int N, int dk, int dv, bool has_state_in, bool has_dstate, bool want_dstate_in) {
  const int share = 148 / 3;
  const int chunk = backward_chunk(N);
  int n = 0;
  if (has_state_in || has_dstate) n += 1;  // starting states
  if (want_dstate_in) n += 1;
  if (has_dstate) n += 1;
  const int w[3][2] = {{dv, dk}, {dv, dk}, {dk, dv}};
  for (int i = 0; i < 3; ++i) {
    const int parts = (w[i][0] + kPartWidth - 1) / kPartWidth;
    for (int j = 0; j < parts; ++j) {
      ChunkPlan plan;
      if (!chunk_tc_plan(B, H, N, std::min(kPartWidth, w[i][0] - j * kPartWidth), w[i][1], chunk, share, &plan))
        return -1;
      n += chunk_tc_launch_count(plan) + (j > 0 ? 1 : 0);  // a part after the first adds its sum
    }
  }
  return n;
}

}  // namespace ret
