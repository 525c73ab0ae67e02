// abi.cu -- the extern "C" entry points declared in include/retention.h:
// argument validation (host only, before anything is enqueued), planning and
// dispatch to the kernels in simt.cu, chunk_tc.cu, backward.cu, rotate.cu and
// groupnorm.cu.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "internal.h"
#include "retention.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Common checks of a sequence call (chunkwise / parallel).  When N == 0 the
// data pointers may be NULL (nothing is read or written).
int check_sequence(const void* q, const void* k, const void* v, const float* gamma, const void* out,
                   const void* state_out, int B, int H, int N, int dk, int dv) {
  if (B <= 0 || H <= 0 || N < 0 || dk <= 0 || dv <= 0) return RET_ERR_INVALID;
  if ((int64_t)B * H > INT32_MAX) return RET_ERR_INVALID;
  if (N > 0) {
    if (!q || !k || !v || !gamma || !out) return RET_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
      return RET_ERR_INVALID;
    if (!aligned(gamma, 4)) return RET_ERR_INVALID;
  }
  if (state_out && !aligned(state_out, 16)) return RET_ERR_INVALID;
  return RET_OK;
}

int check_step(const void* q, const void* k, const void* v, const float* state, const void* out,
               int B, int H, int dk, int dv) {
  if (B <= 0 || H <= 0 || dk <= 0 || dv <= 0) return RET_ERR_INVALID;
  if ((int64_t)B * H > INT32_MAX) return RET_ERR_INVALID;
  if (!q || !k || !v || !state || !out) return RET_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(state, 16) ||
      !aligned(out, 16))
    return RET_ERR_INVALID;
  if (dv % 4 != 0) return RET_ERR_UNSUPPORTED;
  return RET_OK;
}

// A byte range [p, p + bytes) of device memory.
struct Span {
  const void* p;
  size_t bytes;
};
bool overlap(const Span& a, const Span& b) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a.bytes > 0 && b.bytes > 0 && a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? RET_OK : RET_ERR_CUDA; }

// Zero the state of an empty sequence (the sum over no tokens).
int zero_state(float* state_out, int B, int H, int dk, int dv, cudaStream_t s) {
  if (!state_out) return RET_OK;
  return from_cuda(cudaMemsetAsync(state_out, 0, sizeof(float) * (size_t)B * H * dk * dv, s));
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// The bf16 chunkwise plan for these sizes, or an error status.  ws_limit:
// the workspace the caller can give (the last wave's units are cut only if
// their segment states fit).
int plan_chunkwise(int B, int H, int N, int dk, int dv, int chunk, int sms, ret::ChunkPlan* plan,
                   size_t ws_limit = SIZE_MAX, int tile = 0) {
  if (B <= 0 || H <= 0 || N < 0 || dk <= 0 || dv <= 0 || chunk <= 0) return RET_ERR_INVALID;
  if (!ret::chunk_tc_plan(B, H, N, dk, dv, chunk, sms, plan, ws_limit, tile)) return RET_ERR_UNSUPPORTED;
  return RET_OK;
}

// bf16 chunkwise call that allocates its segment-state workspace
// stream-ordered (cudaMallocAsync / cudaFreeAsync on the call's stream).
int chunkwise_alloc(const void* q, const void* k, const void* v, const float* gamma,
                    const float* state_in, void* out, float* state_out, int B, int H, int N, int dk,
                    int dv, int chunk, const ret::ChunkNorm* norm, void* stream,
                    const ret::ChunkRotation* rot = nullptr) {
  int st = check_sequence(q, k, v, gamma, out, state_out, B, H, N, dk, dv);
  if (st != RET_OK) return st;
  ret::ChunkPlan plan;
  const int sms = num_sms();
  if (sms <= 0) return RET_ERR_CUDA;
  st = plan_chunkwise(B, H, N, dk, dv, chunk, sms, &plan);
  if (st != RET_OK) return st;
  // GroupNorm: a head's whole row, unpadded, in one CTA (dv of 64 or 128),
  // with query/key tiles of at most 256 columns
  if (norm && (plan.n_dv_tiles != 1 || plan.dvt != dv || plan.dk_tile > 256)) return RET_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    // the state after no tokens is the state before them
    if (!state_out) return RET_OK;
    if (!state_in) return zero_state(state_out, B, H, dk, dv, s);
    return from_cuda(cudaMemcpyAsync(state_out, state_in, sizeof(float) * (size_t)B * H * dk * dv,
                                     cudaMemcpyDeviceToDevice, s));
  }
  float* ws = nullptr;
  if (plan.workspace_bytes > 0) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&ws), plan.workspace_bytes, s) != cudaSuccess)
      return RET_ERR_CUDA;
  }
  cudaError_t e = ret::launch_chunk_tc(q, k, v, gamma, state_in, out, state_out, B, H, N, dk, dv, plan, ws,
                                       norm, 0.f, s, rot);
  if (ws) {
    cudaError_t e2 = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = e2;
  }
  return from_cuda(e);
}

// Gradients of the forward, bf16 or fp32 tensors (see retention_backward).
int backward_call(bool bf16, const void* q, const void* k, const void* v, const float* gamma,
                  const float* state_in, const void* dout, const float* dstate, void* dq, void* dk_out,
                  void* dv_out, float* dstate_in, int B, int H, int N, int dk, int dv, void* stream) {
  int st = check_sequence(q, k, v, gamma, dout, nullptr, B, H, N, dk, dv);
  if (st != RET_OK) return st;
  if (N > 0) {
    if (!dq || !dk_out || !dv_out) return RET_ERR_INVALID;
    if (!aligned(dq, 16) || !aligned(dk_out, 16) || !aligned(dv_out, 16)) return RET_ERR_INVALID;
  }
  if ((state_in && !aligned(state_in, 16)) || (dstate && !aligned(dstate, 16)) ||
      (dstate_in && !aligned(dstate_in, 16)))
    return RET_ERR_INVALID;
  if (dstate_in && (dstate_in == dstate || dstate_in == state_in)) return RET_ERR_INVALID;
  if (N > 0) {
    // The kernels read q, k, v and dout while other CTAs already write the
    // gradients, so no gradient may overlap an input or another gradient.
    const size_t el = bf16 ? 2 : 4, rows = (size_t)B * H * N;
    const Span in[4] = {{q, rows * dk * el}, {k, rows * dk * el}, {v, rows * dv * el}, {dout, rows * dv * el}};
    const Span outs[3] = {{dq, rows * dk * el}, {dk_out, rows * dk * el}, {dv_out, rows * dv * el}};
    for (int i = 0; i < 3; ++i) {
      for (const Span& x : in)
        if (overlap(outs[i], x)) return RET_ERR_INVALID;
      for (int j = i + 1; j < 3; ++j)
        if (overlap(outs[i], outs[j])) return RET_ERR_INVALID;
    }
  }
  if (dk % 4 != 0 || dv % 4 != 0 || dk > 512 || dv > 512 ||
      ret::backward_smem_bytes(dk, dv) > (size_t)ret::kMaxSmemPerBlock)
    return RET_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    // the gradient reaches the starting state unchanged through no tokens
    if (!dstate_in) return RET_OK;
    if (!dstate) return zero_state(dstate_in, B, H, dk, dv, s);
    return from_cuda(cudaMemcpyAsync(dstate_in, dstate, sizeof(float) * (size_t)B * H * dk * dv,
                                     cudaMemcpyDeviceToDevice, s));
  }
  if (bf16 && ret::backward_tc_supported(dk, dv) && (int64_t)B * H <= 65535)
    return from_cuda(ret::launch_backward_tc(q, k, v, gamma, state_in, dout, dstate, dq, dk_out, dv_out, dstate_in, B,
                                             H, N, dk, dv, s));
  return from_cuda(ret::launch_backward(bf16, q, k, v, gamma, state_in, dout, dstate, dq, dk_out, dv_out,
                                        dstate_in, B, H, N, dk, dv, s));
}

}  // namespace

namespace ret {
// Workspace of the plan a call with at most `limit` bytes of workspace runs.
int chunkwise_workspace_within(int B, int H, int N, int dk, int dv, int chunk, size_t limit, size_t* bytes) {
  if (!bytes) return RET_ERR_INVALID;
  ChunkPlan plan;
  const int sms = num_sms();
  if (sms <= 0) return RET_ERR_CUDA;
  const int st = plan_chunkwise(B, H, N, dk, dv, chunk, sms, &plan, limit);
  if (st != RET_OK) return st;
  *bytes = plan.workspace_bytes;
  return RET_OK;
}
}  // namespace ret

extern "C" {

int retention_version(void) { return 100; }

const char* retention_status_string(int status) {
  switch (status) {
    case RET_OK: return "ok";
    case RET_ERR_INVALID: return "invalid argument";
    case RET_ERR_UNSUPPORTED: return "unsupported shape or chunk size";
    case RET_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int retention_gamma_schedule(int H, float* gamma_out) {
  if (H <= 0 || !gamma_out) return RET_ERR_INVALID;
  for (int h = 0; h < H; ++h) {
    // 1 - 2^(-5-h) rounded once to fp32 ("3. Multi-Scale Retention (MSR)", 0-based h);
    // beyond h = 60 the double value is already 1 - tiny and rounds to 1.0f.
    const double g = h > 60 ? 1.0 : 1.0 - ldexp(1.0, -5 - h);
    gamma_out[h] = (float)g;
  }
  return RET_OK;
}

int retention_test_stall_waits(unsigned int microseconds) {
  if (microseconds > 10000000u) return RET_ERR_INVALID;  // at most 10 s
  ret::g_test_stall_us.store(microseconds, std::memory_order_relaxed);
  return RET_OK;
}

int retention_device_status(unsigned int* flags, int clear) {
  if (!flags) return RET_ERR_INVALID;
  unsigned int a = 0, b = 0;
  cudaError_t e = ret::read_device_status(&a, clear);  // synchronises the device first
  if (e == cudaSuccess) e = ret::read_parallel_status(&b, clear);
  *flags = a | b;
  return from_cuda(e);
}

int retention_chunkwise_workspace_size(int B, int H, int N, int dk, int dv, int chunk,
                                       size_t* bytes) {
  if (!bytes) return RET_ERR_INVALID;
  ret::ChunkPlan plan;
  const int sms = num_sms();
  int st = plan_chunkwise(B, H, N, dk, dv, chunk, sms > 0 ? sms : 148, &plan);
  if (st != RET_OK) return st;
  *bytes = plan.workspace_bytes;
  return RET_OK;
}

int retention_chunkwise_launches(int B, int H, int N, int dk, int dv, int chunk, int* launches) {
  if (!launches) return RET_ERR_INVALID;
  ret::ChunkPlan plan;
  const int sms = num_sms();
  int st = plan_chunkwise(B, H, N, dk, dv, chunk, sms > 0 ? sms : 148, &plan);
  if (st != RET_OK) return st;
  *launches = N == 0 ? 0 : ret::chunk_tc_launch_count(plan);
  return RET_OK;
}

int retention_chunkwise_ws(const void* q, const void* k, const void* v, const float* gamma,
                           void* out, float* state_out, int B, int H, int N, int dk, int dv,
                           int chunk, void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_sequence(q, k, v, gamma, out, state_out, B, H, N, dk, dv);
  if (st != RET_OK) return st;
  ret::ChunkPlan plan;
  const int sms = num_sms();
  if (sms <= 0) return RET_ERR_CUDA;
  st = plan_chunkwise(B, H, N, dk, dv, chunk, sms, &plan, workspace ? workspace_bytes : 0);
  if (st != RET_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) return zero_state(state_out, B, H, dk, dv, s);
  if (plan.workspace_bytes > 0) {
    if (!workspace || workspace_bytes < plan.workspace_bytes || !aligned(workspace, 256))
      return RET_ERR_INVALID;
  }
  return from_cuda(ret::launch_chunk_tc(q, k, v, gamma, nullptr, out, state_out, B, H, N, dk, dv, plan,
                                        static_cast<float*>(workspace), nullptr, 0.f, s));
}

int retention_chunkwise(const void* q, const void* k, const void* v, const float* gamma, void* out,
                        float* state_out, int B, int H, int N, int dk, int dv, int chunk,
                        void* stream) {
  return chunkwise_alloc(q, k, v, gamma, nullptr, out, state_out, B, H, N, dk, dv, chunk, nullptr, stream);
}

int retention_chunkwise_from_state(const void* q, const void* k, const void* v, const float* gamma,
                                   const float* state_in, void* out, float* state_out, int B, int H,
                                   int N, int dk, int dv, int chunk, void* stream) {
  if (state_in && (!aligned(state_in, 16) || state_in == state_out)) return RET_ERR_INVALID;
  return chunkwise_alloc(q, k, v, gamma, state_in, out, state_out, B, H, N, dk, dv, chunk, nullptr, stream);
}

int retention_chunkwise_rotated(const void* q, const void* k, const void* v, const float* gamma, const float* theta,
                                int n0, const float* state_in, void* out, float* state_out, int B, int H, int N,
                                int dk, int dv, int chunk, void* stream) {
  if (!theta || !aligned(theta, 4) || n0 < 0) return RET_ERR_INVALID;
  if (state_in && (!aligned(state_in, 16) || state_in == state_out)) return RET_ERR_INVALID;
  // every row of every tile, padding included, at an exact float position
  const int tile = chunk == 32 ? 64 : chunk;
  if (chunk > 0 && N >= 0 && (int64_t)n0 + ((int64_t)N + tile - 1) / tile * tile > (1 << 24))
    return RET_ERR_UNSUPPORTED;
  const ret::ChunkRotation rot{theta, n0};
  // Where the rotation is fused, the output group turns each Q/K slot in
  // shared memory.  That pays with one value tile per head (mid: 45.7 us
  // against 47.7 us for two rotation passes and the chunkwise call); with
  // several value-tile CTAs per head (each would turn the same Q/K tiles) the
  // extra instructions on that latency-bound group cost more than the HBM
  // traffic they save, so q and k are turned by the standalone pass into
  // scratch first.
  int st = check_sequence(q, k, v, gamma, out, state_out, B, H, N, dk, dv);
  if (st != RET_OK) return st;
  ret::ChunkPlan plan;
  const int sms = num_sms();
  if (sms <= 0) return RET_ERR_CUDA;
  st = plan_chunkwise(B, H, N, dk, dv, chunk, sms, &plan);
  if (st != RET_OK) return st;
  if (N == 0 || (plan.n_dv_tiles == 1 && plan.dk_tile <= 256))
    return chunkwise_alloc(q, k, v, gamma, state_in, out, state_out, B, H, N, dk, dv, chunk, nullptr, stream, &rot);
  if (!ret::rotate_supported(N, dk, n0)) return RET_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)B * H * N * dk * 2;  // one turned copy of q or k (bf16)
  char* scratch = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&scratch), 2 * bytes, s) != cudaSuccess) return RET_ERR_CUDA;
  cudaError_t e = ret::launch_rotate_bf16(q, theta, scratch, B, H, N, dk, n0, s);
  if (e == cudaSuccess) e = ret::launch_rotate_bf16(k, theta, scratch + bytes, B, H, N, dk, n0, s);
  int r = from_cuda(e);
  if (r == RET_OK)
    r = chunkwise_alloc(scratch, scratch + bytes, v, gamma, state_in, out, state_out, B, H, N, dk, dv, chunk, nullptr,
                        stream);
  const cudaError_t e2 = cudaFreeAsync(scratch, s);
  return r != RET_OK ? r : from_cuda(e2);
}

int retention_chunkwise_groupnorm(const void* q, const void* k, const void* v, const float* gamma,
                                  const float* weight, const float* bias, float eps, void* out,
                                  float* state_out, int B, int H, int N, int dk, int dv, int chunk,
                                  void* stream) {
  if (!(eps >= 0.f) || eps > 1e30f) return RET_ERR_INVALID;  // also rejects NaN
  if ((weight && !aligned(weight, 16)) || (bias && !aligned(bias, 16))) return RET_ERR_INVALID;
  const ret::ChunkNorm norm{weight, bias, eps};
  return chunkwise_alloc(q, k, v, gamma, nullptr, out, state_out, B, H, N, dk, dv, chunk, &norm, stream);
}

int retention_chunkwise_f32(const float* q, const float* k, const float* v, const float* gamma,
                            float* out, float* state_out, int B, int H, int N, int dk, int dv,
                            int chunk, void* stream) {
  int st = check_sequence(q, k, v, gamma, out, state_out, B, H, N, dk, dv);
  if (st != RET_OK) return st;
  if (chunk <= 0) return RET_ERR_INVALID;
  if (chunk > 128 || dk > 256 || dv > 256) return RET_ERR_UNSUPPORTED;
  if (ret::chunkwise_f32_smem_bytes(dk, chunk) > (size_t)ret::kMaxSmemPerBlock)
    return RET_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return from_cuda(ret::launch_chunkwise_f32(q, k, v, gamma, out, state_out, B, H, N, dk, dv,
                                             chunk, s));
}

int retention_rotate(const void* x, const float* theta, void* y, int B, int H, int N, int d, int n0,
                     void* stream) {
  if (B <= 0 || H <= 0 || N < 0 || d <= 0 || n0 < 0) return RET_ERR_INVALID;
  if ((int64_t)B * H > INT32_MAX) return RET_ERR_INVALID;
  if (N > 0) {
    if (!x || !theta || !y || !aligned(x, 16) || !aligned(y, 16) || !aligned(theta, 4))
      return RET_ERR_INVALID;
  }
  if (!ret::rotate_supported(N, d, n0)) return RET_ERR_UNSUPPORTED;
  if (N == 0) return RET_OK;
  return from_cuda(ret::launch_rotate_bf16(x, theta, y, B, H, N, d, n0, static_cast<cudaStream_t>(stream)));
}

int retention_groupnorm(const void* r, const float* weight, const float* bias, void* y, int B, int H,
                        int N, int dv, float eps, void* stream) {
  if (B <= 0 || H <= 0 || N < 0 || dv <= 0) return RET_ERR_INVALID;
  if (!(eps >= 0.f) || eps > 1e30f) return RET_ERR_INVALID;  // also rejects NaN
  if ((int64_t)B * H > INT32_MAX) return RET_ERR_INVALID;
  if (N > 0) {
    if (!r || !y || !aligned(r, 16) || !aligned(y, 16)) return RET_ERR_INVALID;
  }
  if ((weight && !aligned(weight, 4)) || (bias && !aligned(bias, 4))) return RET_ERR_INVALID;
  if (!ret::groupnorm_supported(dv) || (int64_t)B * H > 65535) return RET_ERR_UNSUPPORTED;
  if (N == 0) return RET_OK;
  return from_cuda(ret::launch_groupnorm_bf16(r, weight, bias, y, B, H, N, dv, eps,
                                              static_cast<cudaStream_t>(stream)));
}

int retention_parallel(const void* q, const void* k, const void* v, const float* gamma, void* out,
                       int B, int H, int N, int dk, int dv, void* stream) {
  int st = check_sequence(q, k, v, gamma, out, nullptr, B, H, N, dk, dv);
  if (st != RET_OK) return st;
  if (ret::parallel_tc_supported(dk, dv)) {
    if (N == 0) return RET_OK;
    return from_cuda(ret::launch_parallel_tc(q, k, v, gamma, out, B, H, N, dk, dv, static_cast<cudaStream_t>(stream)));
  }
  if (dk > 256 || dv > 256) return RET_ERR_UNSUPPORTED;
  if (N == 0) return RET_OK;
  if (B * H > 65535) return RET_ERR_UNSUPPORTED;
  return from_cuda(ret::launch_parallel_bf16(q, k, v, gamma, out, B, H, N, dk, dv,
                                             static_cast<cudaStream_t>(stream)));
}

int retention_parallel_f32(const float* q, const float* k, const float* v, const float* gamma,
                           float* out, int B, int H, int N, int dk, int dv, void* stream) {
  int st = check_sequence(q, k, v, gamma, out, nullptr, B, H, N, dk, dv);
  if (st != RET_OK) return st;
  if (dk > 256 || dv > 256) return RET_ERR_UNSUPPORTED;
  if (N == 0) return RET_OK;
  if (B * H > 65535) return RET_ERR_UNSUPPORTED;
  return from_cuda(ret::launch_parallel_f32(q, k, v, gamma, out, B, H, N, dk, dv,
                                            static_cast<cudaStream_t>(stream)));
}

int retention_backward(const void* q, const void* k, const void* v, const float* gamma,
                       const float* state_in, const void* dout, const float* dstate, void* dq, void* dk_out,
                       void* dv_out, float* dstate_in, int B, int H, int N, int dk, int dv, void* stream) {
  return backward_call(true, q, k, v, gamma, state_in, dout, dstate, dq, dk_out, dv_out, dstate_in, B, H, N, dk,
                       dv, stream);
}

int retention_backward_launches(int B, int H, int N, int dk, int dv, int has_state_in, int has_dstate,
                                int want_dstate_in, int* launches) {
  if (!launches || B <= 0 || H <= 0 || N < 0 || dk <= 0 || dv <= 0) return RET_ERR_INVALID;
  if (N == 0) {
    *launches = want_dstate_in ? 1 : 0;
    return RET_OK;
  }
  if (!ret::backward_tc_supported(dk, dv) || (int64_t)B * H > 65535) {
    *launches = 1;
    return RET_OK;
  }
  const int n = ret::backward_tc_launches(B, H, N, dk, dv, has_state_in != 0, has_dstate != 0, want_dstate_in != 0);
  if (n < 0) return RET_ERR_UNSUPPORTED;
  *launches = n;
  return RET_OK;
}

int retention_backward_f32(const float* q, const float* k, const float* v, const float* gamma,
                           const float* state_in, const float* dout, const float* dstate, float* dq,
                           float* dk_out, float* dv_out, float* dstate_in, int B, int H, int N, int dk, int dv,
                           void* stream) {
  return backward_call(false, q, k, v, gamma, state_in, dout, dstate, dq, dk_out, dv_out, dstate_in, B, H, N, dk,
                       dv, stream);
}

int retention_step(const void* q, const void* k, const void* v, float* state, void* out, int B,
                   int H, int dk, int dv, void* stream) {
  int st = check_step(q, k, v, state, out, B, H, dk, dv);
  if (st != RET_OK) return st;
  if (dv > 4 * 65535 * 32) return RET_ERR_UNSUPPORTED;
  return from_cuda(ret::launch_step_bf16(q, k, v, state, out, B, H, dk, dv,
                                         static_cast<cudaStream_t>(stream)));
}

int retention_step_rotated(const void* q, const void* k, const void* v, const float* theta, int pos,
                           float* state, void* out, int B, int H, int dk, int dv, void* stream) {
  int st = check_step(q, k, v, state, out, B, H, dk, dv);
  if (st != RET_OK) return st;
  if (!theta || !aligned(theta, 4) || pos < 0) return RET_ERR_INVALID;
  if (pos >= (1 << 24) || dk % 2 != 0) return RET_ERR_UNSUPPORTED;
  if (dv > 4 * 65535 * 32) return RET_ERR_UNSUPPORTED;
  return from_cuda(ret::launch_step_bf16(q, k, v, state, out, B, H, dk, dv, static_cast<cudaStream_t>(stream), theta,
                                         pos));
}

int retention_step_f32(const float* q, const float* k, const float* v, float* state, float* out,
                       int B, int H, int dk, int dv, void* stream) {
  int st = check_step(q, k, v, state, out, B, H, dk, dv);
  if (st != RET_OK) return st;
  if (dv > 4 * 65535 * 32) return RET_ERR_UNSUPPORTED;
  return from_cuda(ret::launch_step_f32(q, k, v, state, out, B, H, dk, dv,
                                        static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
