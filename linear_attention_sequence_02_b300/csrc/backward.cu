// backward.cu -- gradients of retention on CUDA cores (fp32 arithmetic).
//
// "RetNet Guide: Retentive Networks & The Impossible Triangle", section "3. The
// Chunkwise Recurrent Representation ...": the chunkwise form exists so that
// long sequences can be trained; the page prints no gradient.  Differentiating
// the forward with starting state S0 (queries scaled by s = 1/sqrt(dk)),
//
//   out_n = s sum_{m<=n} g^(n-m) (q_n . k_m) v_m + s g^(n+1) q_n S0,
//   S_N   = g^N S0 + sum_m g^(N-1-m) k_m^T v_m,
//
// for the loss <dout, out> + <dS, S_N> and splitting the sums at chunk
// boundaries gives three scans over chunks i (rows j, l inside a chunk of
// L tokens; zeta_j = g^(j+1), xi_j = g^(L-1-j)):
//
//   dq:  forward over chunks, carrying the forward state X = S_{i-1}
//        dq_j = s (sum_{l<=j} g^(j-l) (dout_j . v_l) k_l + zeta_j X dout_j)
//        X <- g^L X + sum_l xi_l k_l^T v_l
//   dk:  backward over chunks, carrying G = dL/dS_i (G = dS after the last)
//        dk_j = s sum_{l>=j} g^(l-j) (dout_l . v_j) q_l + xi_j G v_j
//   dv:  the same backward scan,
//        dv_j = s sum_{l>=j} g^(l-j) (q_l . k_j) dout_l + xi_j k_j G
//   with G <- g^L G + s sum_l zeta_l q_l^T dout_l after each chunk, and
//   dS0 = G after chunk 0.
//
// All three have one shape: rows a_j against rows b_l give the in-chunk
// scores P, which weigh rows w_l (a 32-column slab of the gradient being
// made); a state slab St[t][c] (t over the slab, c over the width of a) adds
// the cross term sum_c St[t][c] a_j[c] and takes a rank-L update from w and b.
//   role   direction  a     b     w     state St[t][c]
//   dq     forward    dout  v     k     X[t][c]  (t over dk, c over dv)
//   dk     backward   v     dout  q     G[t][c]  (t over dk, c over dv)
//   dv     backward   k     q     dout  G[c][t]  (t over dv, c over dk)
// One CTA per (b h, role, 32-column slab) walks the chunks with its slab in
// shared memory; one launch makes every gradient.  The chunk length inside
// the kernel is its own choice (the gradients do not depend on it): 32, which
// costs less arithmetic per token than 64 (the scores, recomputed by every
// slab, grow with the chunk) and keeps the tiles at 60 KB for rows of 128, so
// three CTAs share an SM.
//
// Each chunk is four phases separated by barriers: load (a, b rows row-major,
// the w slab transposed; each thread issues all its global loads before it
// stores any), scores (a 2x2 register tile per thread over float4 loads),
// gradient rows (1x4 per thread), state update (4x4 per thread per 128
// columns).  Rows a thread owns are strided (16 or 8 apart) so that the eight
// lanes of a quarter warp read distinct bank groups.  The phase bodies are
// __host__ __device__ functions of the thread index, so the same code can be
// stepped thread by thread on a CPU.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace ret {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdSlab = 32;  // gradient columns per CTA
constexpr int kBwdChunk = 32; // chunk length inside the kernel
constexpr int kBwdLoadBatch = 4;  // loads a thread has in flight in the load phase

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  const float* gamma;
  const float* state_in;  // S0 [B][H][dk][dv] or null (zero)
  const float* dstate;    // dS [B][H][dk][dv] or null (zero)
  void* grad_q;
  void* grad_k;
  void* grad_v;
  float* dstate_in;       // dS0 [B][H][dk][dv] or null (not written)
  int H, N, dk, dv;
  int slabs_k, slabs_v;   // ceil(dk / 32), ceil(dv / 32)
  int wmax;               // max(dk, dv)
};

__host__ __device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }

__host__ __device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__host__ __device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__host__ __device__ __forceinline__ void st1(float* p, float x) { *p = x; }
__host__ __device__ __forceinline__ void st1(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
__host__ __device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}

// What one CTA computes.
struct BwdRole {
  int role;   // 0: dq, 1: dk, 2: dv
  bool fwd;   // forward over chunks (dq) or backward
  int t0;     // first gradient column of the slab
  int nt;     // valid columns in the slab (a multiple of 4)
  int wa;     // width of a and b rows (contracted), of the state rows
  int wo;     // width of w rows and of the gradient rows
  size_t bh;
  float g, scale;
};

__host__ __device__ inline BwdRole bwd_role(const BwdArgs& p, int bx, int by) {
  BwdRole r;
  int slab = by;
  if (slab < p.slabs_k) {
    r.role = 0;
  } else if (slab < 2 * p.slabs_k) {
    r.role = 1;
    slab -= p.slabs_k;
  } else {
    r.role = 2;
    slab -= 2 * p.slabs_k;
  }
  r.fwd = r.role == 0;
  r.t0 = slab * kBwdSlab;
  r.wa = r.role == 2 ? p.dk : p.dv;
  r.wo = r.role == 2 ? p.dv : p.dk;
  r.nt = imin(kBwdSlab, r.wo - r.t0);
  r.bh = (size_t)bx;
  r.g = p.gamma[bx % p.H];
  r.scale = 1.0f / sqrtf((float)p.dk);
  return r;
}

// Shared-memory regions (floats; every region starts on a 16-byte boundary).
template <int C>
struct BwdSmem {
  float* As;  // [C][lda]     a rows
  float* Bs;  // [C][lda]     b rows
  float* WT;  // [32][C + 4]  w slab, transposed: WT[t][l]
  float* P;   // [C][C + 4]   scores
  float* St;  // [32][lda]    state slab
  float* pw;  // [C + 4]      g^0 .. g^C
  int lda;    // wmax + 4
  static constexpr int ldp = C + 4;
  __host__ __device__ static size_t floats(int wmax) {
    const size_t lda = (size_t)wmax + 4;
    return 2 * C * lda + kBwdSlab * (size_t)ldp + (size_t)C * ldp + kBwdSlab * lda + C + 4;
  }
  __host__ __device__ BwdSmem(float* base, int wmax) {
    lda = wmax + 4;
    As = base;
    Bs = As + (size_t)C * lda;
    WT = Bs + (size_t)C * lda;
    P = WT + (size_t)kBwdSlab * ldp;
    St = P + (size_t)C * ldp;
    pw = St + (size_t)kBwdSlab * lda;
  }
};

// g^d table and the starting state slab: dq starts from S0, dk and dv from dS.
template <int C>
__host__ __device__ inline void bwd_init(const BwdArgs& p, const BwdRole& r, const BwdSmem<C>& s, int tid) {
  const float lg = r.g > 0.f ? log2f(r.g) : 0.f;
  for (int d = tid; d <= C; d += kBwdThreads) s.pw[d] = d == 0 ? 1.f : (r.g > 0.f ? exp2f((float)d * lg) : 0.f);
  const float* src = r.fwd ? p.state_in : p.dstate;
  if (src) src += r.bh * (size_t)p.dk * p.dv;
  const int w4 = r.wa / 4;
  for (int e = tid; e < kBwdSlab * w4; e += kBwdThreads) {
    const int t = e / w4, c = 4 * (e % w4);
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (src && t < r.nt) {
      if (r.role == 2) {
        const float* col = src + (size_t)c * p.dv + r.t0 + t;
        x = make_float4(col[0], col[p.dv], col[2 * (size_t)p.dv], col[3 * (size_t)p.dv]);
      } else {
        x = ld4(src + (size_t)(r.t0 + t) * p.dv + c);
      }
    }
    *reinterpret_cast<float4*>(s.St + (size_t)t * s.lda + c) = x;
  }
}

// a, b rows of the chunk row-major; the w slab transposed; rows and columns
// from L up to the chunk length are zero.
template <int C, typename T>
__host__ __device__ inline void bwd_load(const BwdArgs& p, const BwdRole& r, const BwdSmem<C>& s, int s0, int L,
                                         int tid) {
  const T* Q = static_cast<const T*>(p.q) + r.bh * (size_t)p.N * p.dk;
  const T* K = static_cast<const T*>(p.k) + r.bh * (size_t)p.N * p.dk;
  const T* V = static_cast<const T*>(p.v) + r.bh * (size_t)p.N * p.dv;
  const T* DO = static_cast<const T*>(p.dout) + r.bh * (size_t)p.N * p.dv;
  const T* A = r.role == 0 ? DO : (r.role == 1 ? V : K);
  const T* Bm = r.role == 0 ? V : (r.role == 1 ? DO : Q);
  const T* W = r.role == 0 ? K : (r.role == 1 ? Q : DO);
  const int w4 = r.wa / 4;
  for (int e0 = tid; e0 < C * w4; e0 += kBwdLoadBatch * kBwdThreads) {
    float4 a[kBwdLoadBatch], b[kBwdLoadBatch];
#pragma unroll
    for (int u = 0; u < kBwdLoadBatch; ++u) {
      const int e = e0 + u * kBwdThreads;
      const int j = e / w4, c = 4 * (e % w4);
      a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < C * w4 && j < L) {
        a[u] = ld4(A + (size_t)(s0 + j) * r.wa + c);
        b[u] = ld4(Bm + (size_t)(s0 + j) * r.wa + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kBwdLoadBatch; ++u) {
      const int e = e0 + u * kBwdThreads;
      const int j = e / w4, c = 4 * (e % w4);
      if (e < C * w4) {
        *reinterpret_cast<float4*>(s.As + (size_t)j * s.lda + c) = a[u];
        *reinterpret_cast<float4*>(s.Bs + (size_t)j * s.lda + c) = b[u];
      }
    }
  }
  for (int e = tid; e < C * (kBwdSlab / 4); e += kBwdThreads) {
    const int l = e / (kBwdSlab / 4), t = 4 * (e % (kBwdSlab / 4));
    float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
    if (l < L && t < r.nt) w = ld4(W + (size_t)(s0 + l) * r.wo + r.t0 + t);
    s.WT[(t + 0) * s.ldp + l] = w.x;
    s.WT[(t + 1) * s.ldp + l] = w.y;
    s.WT[(t + 2) * s.ldp + l] = w.z;
    s.WT[(t + 3) * s.ldp + l] = w.w;
  }
}

// P[j][l] = g^|j-l| a_j . b_l on the causal side (l <= j forward, l >= j
// backward) inside the chunk, else 0.  Thread: rows j = tj + 16x, l = tl + 16y.
// Since |tj - tl| < 16, the pairs with y > x (forward) or y < x (backward)
// are always on the masked side: they are written as 0 without a product.
template <int C, bool FWD>
__host__ __device__ inline void bwd_scores(const BwdSmem<C>& s, int wa, int L, int tid) {
  constexpr int M = C / 16;
  const int tj = tid / 16, tl = tid % 16;
  float acc[M][M];
#pragma unroll
  for (int x = 0; x < M; ++x)
#pragma unroll
    for (int y = 0; y < M; ++y) acc[x][y] = 0.f;
  for (int c = 0; c < wa; c += 4) {
    float4 a[M], b[M];
#pragma unroll
    for (int x = 0; x < M; ++x) a[x] = ld4(s.As + (size_t)(tj + 16 * x) * s.lda + c);
#pragma unroll
    for (int y = 0; y < M; ++y) b[y] = ld4(s.Bs + (size_t)(tl + 16 * y) * s.lda + c);
#pragma unroll
    for (int x = 0; x < M; ++x)
#pragma unroll
      for (int y = 0; y < M; ++y)
        if (FWD ? y <= x : y >= x) acc[x][y] = dot4(a[x], b[y], acc[x][y]);
  }
#pragma unroll
  for (int x = 0; x < M; ++x)
#pragma unroll
    for (int y = 0; y < M; ++y) {
      const int j = tj + 16 * x, l = tl + 16 * y;
      const bool keep = j < L && l < L && (FWD ? l <= j : l >= j);
      s.P[j * s.ldp + l] = keep ? s.pw[FWD ? j - l : l - j] * acc[x][y] : 0.f;
    }
}

template <int C>
__host__ __device__ inline void bwd_scores(const BwdRole& r, const BwdSmem<C>& s, int L, int tid) {
  if (r.fwd)
    bwd_scores<C, true>(s, r.wa, L, tid);
  else
    bwd_scores<C, false>(s, r.wa, L, tid);
}

// Gradient rows: in-chunk sum over P and the w slab, plus the cross term of a
// with the state slab.  Thread: rows j = rj + 32y, columns t = rt + 8x.
template <int C, typename T>
__host__ __device__ inline void bwd_rows(const BwdArgs& p, const BwdRole& r, const BwdSmem<C>& s, int s0, int L,
                                         int tid) {
  constexpr int MY = C / 32;
  const int rj = tid / 8, rt = tid % 8;
  const int Lr = (L + 3) & ~3;
  // P is zero off the causal side, so the inner sum runs over the 4-column
  // groups that hold l <= j (forward) or l >= j (backward) for this thread's j
  const int l_begin = r.fwd ? 0 : (rj & ~3);
  const int l_end = r.fwd ? imin(Lr, ((rj + 32 * (MY - 1)) | 3) + 1) : Lr;
  float inner[MY][4], cross[MY][4];
#pragma unroll
  for (int y = 0; y < MY; ++y)
#pragma unroll
    for (int x = 0; x < 4; ++x) inner[y][x] = cross[y][x] = 0.f;
  for (int l = l_begin; l < l_end; l += 4) {
    float4 pj[MY], wt[4];
#pragma unroll
    for (int y = 0; y < MY; ++y) pj[y] = ld4(s.P + (rj + 32 * y) * s.ldp + l);
#pragma unroll
    for (int x = 0; x < 4; ++x) wt[x] = ld4(s.WT + (rt + 8 * x) * s.ldp + l);
#pragma unroll
    for (int y = 0; y < MY; ++y)
#pragma unroll
      for (int x = 0; x < 4; ++x) inner[y][x] = dot4(pj[y], wt[x], inner[y][x]);
  }
  for (int c = 0; c < r.wa; c += 4) {
    float4 aj[MY], st[4];
#pragma unroll
    for (int y = 0; y < MY; ++y) aj[y] = ld4(s.As + (size_t)(rj + 32 * y) * s.lda + c);
#pragma unroll
    for (int x = 0; x < 4; ++x) st[x] = ld4(s.St + (size_t)(rt + 8 * x) * s.lda + c);
#pragma unroll
    for (int y = 0; y < MY; ++y)
#pragma unroll
      for (int x = 0; x < 4; ++x) cross[y][x] = dot4(aj[y], st[x], cross[y][x]);
  }
  T* Out = static_cast<T*>(r.role == 0 ? p.grad_q : (r.role == 1 ? p.grad_k : p.grad_v)) + r.bh * (size_t)p.N * r.wo;
#pragma unroll
  for (int y = 0; y < MY; ++y) {
    const int j = rj + 32 * y;
    if (j >= L) continue;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int t = rt + 8 * x;
      if (t >= r.nt) continue;
      const float v = r.fwd ? r.scale * (inner[y][x] + s.pw[j + 1] * cross[y][x])
                            : fmaf(r.scale, inner[y][x], s.pw[L - 1 - j] * cross[y][x]);
      st1(Out + (size_t)(s0 + j) * r.wo + r.t0 + t, v);
    }
  }
}

// State slab: St = g^L St + sum_l coef_l w_l^T b_l, coef_l = g^(L-1-l)
// forward, s g^(l+1) backward.  Thread: rows t = ut + 8x, columns 4 (ug + 32k).
template <int C>
__host__ __device__ inline void bwd_update(const BwdRole& r, const BwdSmem<C>& s, int L, int tid) {
  const int ut = tid % 8, ug = tid / 8;
  const int Lr = (L + 3) & ~3;
  const float gL = s.pw[L];
  for (int c = 4 * ug; c < r.wa; c += 4 * (kBwdThreads / 8)) {
    float4 u[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) u[x] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int l = 0; l < Lr; l += 4) {
      float cf[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int li = l + i;
        cf[i] = li < L ? (r.fwd ? s.pw[L - 1 - li] : r.scale * s.pw[li + 1]) : 0.f;
      }
      float4 b[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) b[i] = ld4(s.Bs + (size_t)(l + i) * s.lda + c);
#pragma unroll
      for (int x = 0; x < 4; ++x) w[x] = ld4(s.WT + (ut + 8 * x) * s.ldp + l);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float wx[4] = {cf[0] * w[x].x, cf[1] * w[x].y, cf[2] * w[x].z, cf[3] * w[x].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          u[x].x = fmaf(wx[i], b[i].x, u[x].x);
          u[x].y = fmaf(wx[i], b[i].y, u[x].y);
          u[x].z = fmaf(wx[i], b[i].z, u[x].z);
          u[x].w = fmaf(wx[i], b[i].w, u[x].w);
        }
      }
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      float4* sp = reinterpret_cast<float4*>(s.St + (size_t)(ut + 8 * x) * s.lda + c);
      const float4 o = *sp;
      *sp = make_float4(fmaf(gL, o.x, u[x].x), fmaf(gL, o.y, u[x].y), fmaf(gL, o.z, u[x].z), fmaf(gL, o.w, u[x].w));
    }
  }
}

// dS0: the dk role's slab holds rows t0.. of G after chunk 0.
template <int C>
__host__ __device__ inline void bwd_final(const BwdArgs& p, const BwdRole& r, const BwdSmem<C>& s, int tid) {
  if (r.role != 1 || !p.dstate_in) return;
  float* dst = p.dstate_in + r.bh * (size_t)p.dk * p.dv;
  const int w4 = p.dv / 4;
  for (int e = tid; e < r.nt * w4; e += kBwdThreads) {
    const int t = e / w4, c = 4 * (e % w4);
    *reinterpret_cast<float4*>(dst + (size_t)(r.t0 + t) * p.dv + c) = ld4(s.St + (size_t)t * s.lda + c);
  }
}

template <int C, typename T>
__global__ void __launch_bounds__(kBwdThreads, 3) backward_kernel(BwdArgs p) {
  extern __shared__ float4 sm4[];
  const BwdRole r = bwd_role(p, blockIdx.x, blockIdx.y);
  const BwdSmem<C> s(reinterpret_cast<float*>(sm4), p.wmax);
  const int tid = threadIdx.x;
  bwd_init<C>(p, r, s, tid);
  const int n_chunks = (p.N + C - 1) / C;
  for (int it = 0; it < n_chunks; ++it) {
    const int s0 = (r.fwd ? it : n_chunks - 1 - it) * C;
    const int L = imin(C, p.N - s0);
    __syncthreads();  // the previous chunk's tiles are consumed; pw and St are written
    bwd_load<C, T>(p, r, s, s0, L, tid);
    __syncthreads();
    bwd_scores<C>(r, s, L, tid);
    __syncthreads();
    bwd_rows<C, T>(p, r, s, s0, L, tid);
    __syncthreads();  // the rows have read the state slab
    bwd_update<C>(r, s, L, tid);
  }
  __syncthreads();
  bwd_final<C>(p, r, s, tid);
}

template <int C, typename T>
cudaError_t launch_bwd(const BwdArgs& a, int BH, cudaStream_t s) {
  const size_t smem = sizeof(float) * BwdSmem<C>::floats(a.wmax);
  cudaError_t e = cudaFuncSetAttribute(backward_kernel<C, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)BH, (unsigned)(2 * a.slabs_k + a.slabs_v));
  backward_kernel<C, T><<<grid, kBwdThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int backward_chunk(int, int) { return kBwdChunk; }

size_t backward_smem_bytes(int dk, int dv) {
  return sizeof(float) * BwdSmem<kBwdChunk>::floats(dk > dv ? dk : dv);
}

cudaError_t launch_backward(bool bf16, const void* q, const void* k, const void* v, const float* gamma,
                            const float* state_in, const void* dout, const float* dstate, void* dq, void* dk_out,
                            void* dv_out, float* dstate_in, int B, int H, int N, int dk, int dv, cudaStream_t s) {
  BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.dout = dout;
  a.gamma = gamma;
  a.state_in = state_in;
  a.dstate = dstate;
  a.grad_q = dq;
  a.grad_k = dk_out;
  a.grad_v = dv_out;
  a.dstate_in = dstate_in;
  a.H = H;
  a.N = N;
  a.dk = dk;
  a.dv = dv;
  a.slabs_k = (dk + kBwdSlab - 1) / kBwdSlab;
  a.slabs_v = (dv + kBwdSlab - 1) / kBwdSlab;
  a.wmax = dk > dv ? dk : dv;
  const int BH = B * H;
  return bf16 ? launch_bwd<kBwdChunk, __nv_bfloat16>(a, BH, s) : launch_bwd<kBwdChunk, float>(a, BH, s);
}

}  // namespace ret
