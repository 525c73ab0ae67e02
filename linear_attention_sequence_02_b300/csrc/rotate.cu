// rotate.cu -- the position phase rotation of queries and keys.
//
// "RetNet Guide: Retentive Networks & The Impossible Triangle", section "2.
// Relative Position via Complex Exponential Phase Rotations": the query and key
// of token n carry the phase e^(i n theta), so that their product depends on
// n - m only.  Pairs (2j, 2j+1) of the d real dimensions are one complex
// coordinate with frequency theta_j; with the real dot product of the
// retention kernels, query and key are both turned by the angle (n0 + n)
// theta_j:
//
//   y[2j]   = x[2j] cos a - x[2j+1] sin a,   y[2j+1] = x[2j] sin a + x[2j+1] cos a,
//   a = (n0 + n) theta_j
//
// x, y: bf16 [B][H][N][d] (y may be x).  A thread owns one 16-byte chunk (four
// pairs) of one token: it computes the four angles once and applies them to
// the same chunk of several (b, h) rows, so the sines and cosines are shared
// across heads.  Angles are reduced modulo 2 pi before sincosf by the method
// of Cody and Waite, with the product (n0 + n) theta_j first split exactly into
// two floats, so positions up to 2^24 keep ~1e-7 rad of angle accuracy in
// fp32.  The kernel is bound by HBM: 4 d bytes per row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "angle.cuh"
#include "internal.h"

namespace ret {
namespace {

constexpr int kRotThreads = 256;
constexpr int kRotInFlight = 8;  // (b, h) rows a thread loads before it rotates any

__global__ void __launch_bounds__(kRotThreads)
rotate_kernel(const __nv_bfloat16* x, const float* __restrict__ theta, __nv_bfloat16* y, int BH, int N, int d,
              int n0, int rows_per_cta) {
  const int chunks = d / 8;
  const int t = blockIdx.x * kRotThreads + threadIdx.x;  // token n, chunk c8
  if (t >= N * chunks) return;
  const int n = t / chunks, c8 = t - n * chunks;
  const int bh0 = blockIdx.y * rows_per_cta;
  const int bh1 = min(BH, bh0 + rows_per_cta);
  const size_t row = (size_t)N * d;  // elements between (b, h) rows
  const size_t off = (size_t)n * d + 8 * c8;
  for (int bh = bh0; bh < bh1; bh += kRotInFlight) {
    // the loads first, so their latency overlaps the angles (first batch) or
    // the previous batch's stores
    uint4 v[kRotInFlight];
#pragma unroll
    for (int u = 0; u < kRotInFlight; ++u)
      if (bh + u < bh1) v[u] = *reinterpret_cast<const uint4*>(x + (size_t)(bh + u) * row + off);
    float cs[4], sn[4];
    const float p = (float)(n0 + n);
#pragma unroll
    for (int e = 0; e < 4; ++e) sincosf(reduced_angle(p, __ldg(theta + 4 * c8 + e)), &sn[e], &cs[e]);
#pragma unroll
    for (int u = 0; u < kRotInFlight; ++u) {
      if (bh + u < bh1) {
        const uint4 o = make_uint4(rot_pair(v[u].x, cs[0], sn[0]), rot_pair(v[u].y, cs[1], sn[1]),
                                   rot_pair(v[u].z, cs[2], sn[2]), rot_pair(v[u].w, cs[3], sn[3]));
        *reinterpret_cast<uint4*>(y + (size_t)(bh + u) * row + off) = o;
      }
    }
  }
}

}  // namespace

bool rotate_supported(int N, int d, int n0) {
  return d > 0 && d % 8 == 0 && n0 >= 0 && (int64_t)n0 + N <= (1 << 24) &&
         (int64_t)N * (d / 8) < (int64_t)1 << 31;
}

cudaError_t launch_rotate_bf16(const void* x, const float* theta, void* y, int B, int H, int N, int d,
                               int n0, cudaStream_t s) {
  const int BH = B * H;
  if (BH == 0 || N == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long gx = ((long long)N * (d / 8) + kRotThreads - 1) / kRotThreads;
  // about four CTAs per SM in all: split the (b, h) rows over blockIdx.y, a
  // multiple of the rows a thread has in flight
  long long rows = (BH * gx + 4LL * sms - 1) / (4LL * sms);
  rows = (rows + kRotInFlight - 1) / kRotInFlight * kRotInFlight;
  if (rows < 1) rows = 1;
  if (rows > BH) rows = BH;
  const long long gy = (BH + rows - 1) / rows;
  if (gx > 0x7fffffffLL || gy > 65535) return cudaErrorInvalidConfiguration;
  rotate_kernel<<<dim3((unsigned)gx, (unsigned)gy), kRotThreads, 0, s>>>(
      static_cast<const __nv_bfloat16*>(x), theta, static_cast<__nv_bfloat16*>(y), BH, N, d, n0, (int)rows);
  return cudaGetLastError();
}

}  // namespace ret
