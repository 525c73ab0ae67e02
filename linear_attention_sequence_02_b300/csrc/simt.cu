// simt.cu -- CUDA-core kernels of the retention library:
//   * the recurrent decode step (bf16 and fp32 q/k/v/out, fp32 state in place),
//     an HBM-bound streaming read-modify-write of the state;
//   * the parallel form (bf16 and fp32), tiled over 64x64 output blocks;
//   * the chunkwise form with fp32 inputs (plain fp32 FMA, no TF32).
//
// Formulas follow "RetNet Guide: Retentive Networks & The Impossible
// Triangle": sections "1. The Parallel Representation ..." (D and
// R = ((QK^T) (.) D) V), "2. The Recurrent Representation ..."
// (S_n = gamma S_{n-1} + K_n^T V_n, R_n = Q_n S_n) and "3. The Chunkwise
// Recurrent Representation ..." (chunk carry, zeta_j = gamma^(j+1)); the query
// is divided by sqrt(dk) ("1. PyTorch Implementation of MultiScaleRetention").
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "angle.cuh"
#include "internal.h"

namespace ret {
namespace {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Four consecutive elements as float (16-byte fp32 or 8-byte bf16 load).
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  uint2 raw = *reinterpret_cast<const uint2*>(p);
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
  float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}

// gamma^d for an integer distance d >= 0, with gamma in [0, 1]:
// 1 at d == 0 (also for gamma == 0), else exp2(d * log2(gamma)).
__device__ __forceinline__ float decay_pow(float g, float lg, int d) {
  if (d == 0) return 1.0f;
  if (g <= 0.0f) return 0.0f;
  return exp2f((float)d * lg);
}

// ----------------------------------------------------------------------------
// Decode step.  One CTA of 256 threads (8 warps) per (b*H + h, 128-column
// slab of dv).  Lane l of every warp owns columns c0 = slab*128 + 4l .. +3;
// warp w walks rows w, w+8, ...; each row access is one coalesced 512-byte
// float4 read and write of the state.  Eight rows are loaded before any is
// written so that eight 16-byte loads per thread are in flight.  The column
// partial sums of q~ . S' are reduced across the 8 warps in shared memory.
// gamma_h = 1 - 2^(-5-h) is formed exactly in fp32 from the head index.
// With a rotation (theta non-null), q and k are first turned by the token's
// position ("2. Relative Position via Complex Exponential Phase Rotations":
// pair (2j, 2j+1) by pos theta_j, the angle reduced modulo 2 pi by the method
// of Cody and Waite), in fp32, as they are loaded.
constexpr int kStepThreads = 256;
constexpr int kStepCols = 128;
constexpr int kStepUnroll = 8;

template <typename T>
__global__ void __launch_bounds__(kStepThreads)
step_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
            float* __restrict__ state, T* __restrict__ out, int H, int dk, int dv,
            const float* __restrict__ theta, int pos) {
  extern __shared__ float sm[];
  float* qs = sm;               // [dk]  q / sqrt(dk)
  float* ks = sm + dk;          // [dk]
  float* red = sm + 2 * dk;     // [8][128]
  const int bh = blockIdx.x;
  const int h = bh % H;
  const float g = 1.0f - ldexpf(1.0f, -5 - h);
  const float scale = 1.0f / sqrtf((float)dk);
  if (theta == nullptr) {
    for (int i = threadIdx.x; i < dk; i += kStepThreads) {
      qs[i] = to_f32(q[(size_t)bh * dk + i]) * scale;
      ks[i] = to_f32(k[(size_t)bh * dk + i]);
    }
  } else {
    for (int j = threadIdx.x; 2 * j < dk; j += kStepThreads) {
      float sn, cs;
      sincosf(reduced_angle((float)pos, __ldg(theta + j)), &sn, &cs);
      const float q0 = to_f32(q[(size_t)bh * dk + 2 * j]), q1 = to_f32(q[(size_t)bh * dk + 2 * j + 1]);
      const float k0 = to_f32(k[(size_t)bh * dk + 2 * j]), k1 = to_f32(k[(size_t)bh * dk + 2 * j + 1]);
      qs[2 * j] = (q0 * cs - q1 * sn) * scale;
      qs[2 * j + 1] = (q0 * sn + q1 * cs) * scale;
      ks[2 * j] = k0 * cs - k1 * sn;
      ks[2 * j + 1] = k0 * sn + k1 * cs;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.y * kStepCols + lane * 4;
  const bool active = c0 < dv;  // dv % 4 == 0, so c0+3 < dv too
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (active) {
    const float4 vv = load4(v + (size_t)bh * dv + c0);
    float* S = state + (size_t)bh * dk * dv + c0;
    for (int r0 = warp; r0 < dk; r0 += 8 * kStepUnroll) {
      float4 s[kStepUnroll];
#pragma unroll
      for (int u = 0; u < kStepUnroll; ++u) {
        const int r = r0 + 8 * u;
        if (r < dk) s[u] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)r * dv));
      }
#pragma unroll
      for (int u = 0; u < kStepUnroll; ++u) {
        const int r = r0 + 8 * u;
        if (r < dk) {
          const float kr = ks[r], qr = qs[r];
          float4 t = s[u];
          t.x = fmaf(g, t.x, kr * vv.x);
          t.y = fmaf(g, t.y, kr * vv.y);
          t.z = fmaf(g, t.z, kr * vv.z);
          t.w = fmaf(g, t.w, kr * vv.w);
          __stcs(reinterpret_cast<float4*>(S + (size_t)r * dv), t);
          acc.x = fmaf(qr, t.x, acc.x);
          acc.y = fmaf(qr, t.y, acc.y);
          acc.z = fmaf(qr, t.z, acc.z);
          acc.w = fmaf(qr, t.w, acc.w);
        }
      }
    }
  }
  *reinterpret_cast<float4*>(red + warp * kStepCols + lane * 4) = acc;
  __syncthreads();
  if (threadIdx.x < kStepCols) {
    const int c = blockIdx.y * kStepCols + threadIdx.x;
    if (c < dv) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kStepThreads / 32; ++w) sum += red[w * kStepCols + threadIdx.x];
      out[(size_t)bh * dv + c] = from_f32<T>(sum);
    }
  }
}

template <typename T>
cudaError_t launch_step(const T* q, const T* k, const T* v, float* state, T* out, int B, int H,
                        int dk, int dv, cudaStream_t s, const float* theta = nullptr, int pos = 0) {
  const size_t smem = sizeof(float) * (2 * (size_t)dk + 8 * kStepCols);
  auto kern = step_kernel<T>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((unsigned)(B * H), (unsigned)((dv + kStepCols - 1) / kStepCols));
  kern<<<grid, kStepThreads, smem, s>>>(q, k, v, state, out, H, dk, dv, theta, pos);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// Parallel form.  One CTA per (64-row block of n, b*H + h, 64-column block of
// dv).  For each 64-row block of m up to the diagonal: scores
// P[m][n] = D[n][m] * (q_n . k_m) / sqrt(dk) for the 64x64 tile (D from the
// absolute distance n - m, never factored into gamma^n * gamma^-m), then
// O[n][c] += sum_m P[m][n] v[m][c].  Each thread owns a 4x4 micro-tile.
constexpr int kParT = 64;
constexpr int kParLd = 68;  // padded row length of the transposed tiles

template <typename T>
__global__ void __launch_bounds__(256)
parallel_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                const float* __restrict__ gamma, T* __restrict__ out, int H, int N, int dk,
                int dv) {
  extern __shared__ float sm[];
  float* Qs = sm;                       // [dk][kParLd]  Qs[i][n]
  float* Ks = Qs + (size_t)dk * kParLd; // [dk][kParLd]  Ks[i][m]
  float* Vs = Ks + (size_t)dk * kParLd; // [64][64]      Vs[m][c]
  float* Ps = Vs + kParT * kParT;       // [64][kParLd]  Ps[m][n]
  const int n0 = blockIdx.x * kParT;
  const size_t bh = blockIdx.y;
  const int c0 = blockIdx.z * kParT;
  const int h = (int)(bh % H);
  const float g = gamma[h];
  const float lg = g > 0.f ? log2f(g) : 0.f;
  const float scale = 1.0f / sqrtf((float)dk);
  const T* Q = q + bh * (size_t)N * dk;
  const T* K = k + bh * (size_t)N * dk;
  const T* V = v + bh * (size_t)N * dv;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;

  for (int e = tid; e < dk * kParT; e += 256) {
    const int n = e / dk, i = e % dk;
    Qs[i * kParLd + n] = (n0 + n < N) ? to_f32(Q[(size_t)(n0 + n) * dk + i]) : 0.f;
  }
  float acc[4][4] = {};
  for (int m0 = 0; m0 <= n0 && m0 < N; m0 += kParT) {
    __syncthreads();  // previous tile's Ks/Vs/Ps are no longer read
    for (int e = tid; e < dk * kParT; e += 256) {
      const int m = e / dk, i = e % dk;
      Ks[i * kParLd + m] = (m0 + m < N) ? to_f32(K[(size_t)(m0 + m) * dk + i]) : 0.f;
    }
    for (int e = tid; e < kParT * kParT; e += 256) {
      const int m = e / kParT, c = e % kParT;
      Vs[m * kParT + c] = (m0 + m < N && c0 + c < dv) ? to_f32(V[(size_t)(m0 + m) * dv + c0 + c]) : 0.f;
    }
    __syncthreads();
    // scores for n in ty*4.., m in tx*4..
    float sc[4][4] = {};
    for (int i = 0; i < dk; ++i) {
      const float4 a = *reinterpret_cast<const float4*>(Qs + i * kParLd + ty * 4);
      const float4 b = *reinterpret_cast<const float4*>(Ks + i * kParLd + tx * 4);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) sc[x][y] = fmaf(av[x], bv[y], sc[x][y]);
    }
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int n = n0 + ty * 4 + x, m = m0 + tx * 4 + y;
        const float w = (m <= n) ? decay_pow(g, lg, n - m) * scale * sc[x][y] : 0.f;
        Ps[(tx * 4 + y) * kParLd + ty * 4 + x] = w;
      }
    __syncthreads();
    for (int m = 0; m < kParT; ++m) {
      const float4 p = *reinterpret_cast<const float4*>(Ps + m * kParLd + ty * 4);
      const float4 vv = *reinterpret_cast<const float4*>(Vs + m * kParT + tx * 4);
      const float pv[4] = {p.x, p.y, p.z, p.w}, vvv[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(pv[x], vvv[y], acc[x][y]);
    }
  }
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int n = n0 + ty * 4 + x;
    if (n >= N) continue;
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      const int c = c0 + tx * 4 + y;
      if (c < dv) out[bh * (size_t)N * dv + (size_t)n * dv + c] = from_f32<T>(acc[x][y]);
    }
  }
}

size_t parallel_smem_bytes(int dk) {
  return sizeof(float) * (2 * (size_t)dk * kParLd + kParT * kParT + kParT * kParLd);
}

template <typename T>
cudaError_t launch_parallel(const T* q, const T* k, const T* v, const float* gamma, T* out, int B,
                            int H, int N, int dk, int dv, cudaStream_t s) {
  const size_t smem = parallel_smem_bytes(dk);
  auto kern = parallel_kernel<T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((N + kParT - 1) / kParT), (unsigned)(B * H), (unsigned)((dv + kParT - 1) / kParT));
  kern<<<grid, 256, smem, s>>>(q, k, v, gamma, out, H, N, dk, dv);
  return cudaGetLastError();
}

// ----------------------------------------------------------------------------
// Chunkwise form with fp32 inputs.  One CTA per (b*H + h, 32-column block of
// dv) walks the chunks in order, keeping its 32 state columns in shared
// memory.  Per chunk of L tokens starting at s:
//   P[j][l] = gamma^(j-l) (q_j . k_l)/sqrt(dk)       (l <= j)
//   out[s+j][c] = sum_l P[j][l] v_l[c] + gamma^(j+1) (q_j . S[:,c])/sqrt(dk)
//   S[i][c] = gamma^L S[i][c] + sum_l gamma^(L-1-l) k_l[i] v_l[c]
// The powers gamma^0..gamma^C come from a table built once per CTA.
constexpr int kCwCols = 32;

__global__ void __launch_bounds__(256)
chunkwise_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                     const float* __restrict__ v, const float* __restrict__ gamma,
                     float* __restrict__ out, float* __restrict__ state_out, int H, int N,
                     int dk, int dv, int C) {
  extern __shared__ float sm[];
  const int ldk = dk + 1;
  float* Qc = sm;                          // [C][dk+1]
  float* Kc = Qc + (size_t)C * ldk;        // [C][dk+1]
  float* Vc = Kc + (size_t)C * ldk;        // [C][32]
  float* P = Vc + (size_t)C * kCwCols;     // [C][C]
  float* S = P + (size_t)C * C;            // [dk][32]
  float* pw = S + (size_t)dk * kCwCols;    // [C+1] gamma^d
  const size_t bh = blockIdx.x;
  const int c0 = blockIdx.y * kCwCols;
  const int h = (int)(bh % H);
  const float g = gamma[h];
  const float lg = g > 0.f ? log2f(g) : 0.f;
  const float scale = 1.0f / sqrtf((float)dk);
  const float* Q = q + bh * (size_t)N * dk;
  const float* K = k + bh * (size_t)N * dk;
  const float* V = v + bh * (size_t)N * dv;
  float* O = out + bh * (size_t)N * dv;
  const int tid = threadIdx.x;

  for (int d = tid; d <= C; d += 256) pw[d] = decay_pow(g, lg, d);
  for (int e = tid; e < dk * kCwCols; e += 256) S[e] = 0.f;

  for (int s0 = 0; s0 < N; s0 += C) {
    const int L = min(C, N - s0);
    __syncthreads();  // previous chunk fully consumed; pw/S initialised
    for (int e = tid; e < L * dk; e += 256) {
      const int j = e / dk, i = e % dk;
      Qc[j * ldk + i] = Q[(size_t)(s0 + j) * dk + i];
      Kc[j * ldk + i] = K[(size_t)(s0 + j) * dk + i];
    }
    for (int e = tid; e < L * kCwCols; e += 256) {
      const int j = e / kCwCols, c = e % kCwCols;
      Vc[e] = (c0 + c < dv) ? V[(size_t)(s0 + j) * dv + c0 + c] : 0.f;
    }
    __syncthreads();
    for (int e = tid; e < L * L; e += 256) {
      const int j = e / L, l = e % L;
      float w = 0.f;
      if (l <= j) {
        float d = 0.f;
        for (int i = 0; i < dk; ++i) d = fmaf(Qc[j * ldk + i], Kc[l * ldk + i], d);
        w = pw[j - l] * d * scale;
      }
      P[j * C + l] = w;
    }
    __syncthreads();
    for (int e = tid; e < L * kCwCols; e += 256) {
      const int j = e / kCwCols, c = e % kCwCols;
      float inner = 0.f;
      for (int l = 0; l <= j; ++l) inner = fmaf(P[j * C + l], Vc[l * kCwCols + c], inner);
      float cross = 0.f;
      for (int i = 0; i < dk; ++i) cross = fmaf(Qc[j * ldk + i], S[i * kCwCols + c], cross);
      if (c0 + c < dv) O[(size_t)(s0 + j) * dv + c0 + c] = inner + pw[j + 1] * scale * cross;
    }
    __syncthreads();
    for (int e = tid; e < dk * kCwCols; e += 256) {
      const int i = e / kCwCols, c = e % kCwCols;
      float t = 0.f;
      for (int l = 0; l < L; ++l) t = fmaf(pw[L - 1 - l] * Kc[l * ldk + i], Vc[l * kCwCols + c], t);
      S[e] = fmaf(pw[L], S[e], t);
    }
  }
  __syncthreads();
  if (state_out) {
    float* So = state_out + bh * (size_t)dk * dv;
    for (int e = tid; e < dk * kCwCols; e += 256) {
      const int i = e / kCwCols, c = e % kCwCols;
      if (c0 + c < dv) So[(size_t)i * dv + c0 + c] = S[e];
    }
  }
}

}  // namespace

cudaError_t launch_step_bf16(const void* q, const void* k, const void* v, float* state, void* out,
                             int B, int H, int dk, int dv, cudaStream_t s, const float* theta, int pos) {
  return launch_step(static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                     static_cast<const __nv_bfloat16*>(v), state, static_cast<__nv_bfloat16*>(out),
                     B, H, dk, dv, s, theta, pos);
}

cudaError_t launch_step_f32(const float* q, const float* k, const float* v, float* state,
                            float* out, int B, int H, int dk, int dv, cudaStream_t s) {
  return launch_step(q, k, v, state, out, B, H, dk, dv, s);
}

cudaError_t launch_parallel_bf16(const void* q, const void* k, const void* v, const float* gamma,
                                 void* out, int B, int H, int N, int dk, int dv, cudaStream_t s) {
  return launch_parallel(static_cast<const __nv_bfloat16*>(q),
                         static_cast<const __nv_bfloat16*>(k),
                         static_cast<const __nv_bfloat16*>(v), gamma,
                         static_cast<__nv_bfloat16*>(out), B, H, N, dk, dv, s);
}

cudaError_t launch_parallel_f32(const float* q, const float* k, const float* v,
                                const float* gamma, float* out, int B, int H, int N, int dk,
                                int dv, cudaStream_t s) {
  return launch_parallel(q, k, v, gamma, out, B, H, N, dk, dv, s);
}

size_t chunkwise_f32_smem_bytes(int dk, int chunk) {
  if (dk <= 0 || chunk <= 0) return 0;
  return sizeof(float) * (2 * (size_t)chunk * (dk + 1) + (size_t)chunk * kCwCols +
                          (size_t)chunk * chunk + (size_t)dk * kCwCols + (size_t)chunk + 1);
}

cudaError_t launch_chunkwise_f32(const float* q, const float* k, const float* v,
                                 const float* gamma, float* out, float* state_out, int B, int H,
                                 int N, int dk, int dv, int chunk, cudaStream_t s) {
  const size_t smem = chunkwise_f32_smem_bytes(dk, chunk);
  cudaError_t e = cudaFuncSetAttribute(chunkwise_f32_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(B * H), (unsigned)((dv + kCwCols - 1) / kCwCols));
  chunkwise_f32_kernel<<<grid, 256, smem, s>>>(q, k, v, gamma, out, state_out, H, N, dk, dv, chunk);
  return cudaGetLastError();
}

}  // namespace ret
