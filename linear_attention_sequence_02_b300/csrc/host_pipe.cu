// host_pipe.cu -- retention_chunkwise_host: the chunkwise forward of
// "3. The Chunkwise Recurrent Representation for Ultra-Long Sequence Prefill"
// ("RetNet Guide: Retentive Networks & The Impossible Triangle") for q, k, v
// and outputs in host memory.
//
// The (batch row, head) pairs are cut into slabs of consecutive pairs (whole
// batch rows, or, with one batch row, equal groups of heads).  Each slab is
// copied to the device, run by the chunkwise kernels and copied back on one of
// three streams of the library's own, round robin over three device slots, so
// the host-to-device copy of one slab, the kernels of the previous one and the
// device-to-host copy of the one before overlap (the two copy directions use
// separate copy engines).  The streams are forked from the caller's stream and
// joined back to it with events, so the call is ordered on that stream like
// any other.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "retention.h"

namespace {

constexpr int kSlots = 3;
constexpr int kTargetSlabs = 8;
constexpr int kMaxDevices = 64;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Slabs of `heads` consecutive (b, h) pairs: whole rows (heads = rows * H),
// or with B == 1 a divisor of H.
struct Slabs {
  int heads, count;
  bool whole_rows;
};
Slabs pick_slabs(int B, int H) {
  Slabs s;
  if (B >= 2) {
    const int rows = (B + kTargetSlabs - 1) / kTargetSlabs;
    s.heads = rows * H;
    s.count = (B + rows - 1) / rows;
    s.whole_rows = true;
  } else {
    int d = H;
    for (int c = 1; c <= H; ++c)
      if (H % c == 0 && H / c <= kTargetSlabs) {
        d = c;
        break;
      }
    s.heads = d;
    s.count = H / d;
    s.whole_rows = false;
  }
  return s;
}

// Batch rows, heads per row and first (b, h) pair of slab i.
struct SlabShape {
  int B, H, bh0;
};
SlabShape slab_shape(const Slabs& s, int B, int H, int i) {
  if (s.whole_rows) {
    const int rows = s.heads / H, r0 = i * rows;
    return SlabShape{std::min(rows, B - r0), H, r0 * H};
  }
  return SlabShape{1, s.heads, i * s.heads};
}

// Device bytes of one slot and the offsets of its parts.
struct SlotLayout {
  size_t q, k, v, o, st, ws, bytes, ws_bytes;
};
int slot_layout(int B, int H, int N, int dk, int dv, int chunk, bool want_state, const Slabs& s, int sms,
                SlotLayout* L) {
  const size_t rows = (size_t)s.heads * N;
  size_t ws = 0;
  for (int i = 0; i < s.count; i += std::max(1, s.count - 1)) {  // the first (full) and the last slab
    const SlabShape sh = slab_shape(s, B, H, i);
    ret::ChunkPlan plan;
    if (!ret::chunk_tc_plan(sh.B, sh.H, N, dk, dv, chunk, sms, &plan)) return RET_ERR_UNSUPPORTED;
    ws = std::max(ws, plan.workspace_bytes);
  }
  size_t off = 0;
  L->q = off;
  off += align256(rows * dk * 2);
  L->k = off;
  off += align256(rows * dk * 2);
  L->v = off;
  off += align256(rows * dv * 2);
  L->o = off;
  off += align256(rows * dv * 2);
  L->st = off;
  off += want_state ? align256(sizeof(float) * (size_t)s.heads * dk * dv) : 0;
  L->ws = off;
  off += align256(ws);
  L->ws_bytes = ws;
  L->bytes = off;
  return RET_OK;
}

struct Pipe {
  cudaStream_t st[kSlots];
  cudaEvent_t fork, join[kSlots];
  bool ready;
};
std::mutex g_pipe_lock[kMaxDevices];
Pipe g_pipe[kMaxDevices];

cudaError_t pipe_for(int dev, Pipe** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  Pipe& p = g_pipe[dev];
  if (!p.ready) {
    cudaError_t e = cudaEventCreateWithFlags(&p.fork, cudaEventDisableTiming);
    for (int i = 0; i < kSlots && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&p.st[i], cudaStreamNonBlocking);
    for (int i = 0; i < kSlots && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&p.join[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    p.ready = true;
  }
  *out = &p;
  return cudaSuccess;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? RET_OK : RET_ERR_CUDA; }

}  // namespace

extern "C" {

int retention_chunkwise_host_buffer_size(int B, int H, int N, int dk, int dv, int chunk, size_t* bytes) {
  if (!bytes || B <= 0 || H <= 0 || N < 0 || dk <= 0 || dv <= 0 || chunk <= 0) return RET_ERR_INVALID;
  if ((int64_t)B * H > INT32_MAX) return RET_ERR_INVALID;
  const int sms = sm_count();
  const Slabs s = pick_slabs(B, H);
  SlotLayout L;
  const int st = slot_layout(B, H, std::max(N, 1), dk, dv, chunk, true, s, sms > 0 ? sms : 148, &L);
  if (st != RET_OK) return st;
  *bytes = kSlots * L.bytes;
  return RET_OK;
}

int retention_chunkwise_host(const void* q, const void* k, const void* v, const float* gamma, void* out,
                             float* state_out, int B, int H, int N, int dk, int dv, int chunk, void* dev_buffer,
                             size_t dev_buffer_bytes, void* stream) {
  if (B <= 0 || H <= 0 || N < 0 || dk <= 0 || dv <= 0 || chunk <= 0) return RET_ERR_INVALID;
  if ((int64_t)B * H > INT32_MAX) return RET_ERR_INVALID;
  if (N > 0 && (!q || !k || !v || !gamma || !out)) return RET_ERR_INVALID;
  if (dev_buffer && reinterpret_cast<uintptr_t>(dev_buffer) % 256 != 0) return RET_ERR_INVALID;
  const int sms = sm_count();
  if (sms <= 0) return RET_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RET_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Slabs sl = pick_slabs(B, H);
  SlotLayout L;
  int st = slot_layout(B, H, std::max(N, 1), dk, dv, chunk, state_out != nullptr, sl, sms, &L);
  if (st != RET_OK) return st;
  const size_t need = kSlots * L.bytes;
  if (dev_buffer && dev_buffer_bytes < need) return RET_ERR_INVALID;
  const size_t st_row = sizeof(float) * (size_t)dk * dv;
  if (N == 0) {
    // the state after no tokens is zero
    if (!state_out) return RET_OK;
    const size_t n = st_row * (size_t)B * H;
    void* z = dev_buffer;
    cudaError_t e = cudaSuccess;
    if (!z) e = cudaMallocAsync(&z, n, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(z, 0, n, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(state_out, z, n, cudaMemcpyDeviceToHost, s);
    if (!dev_buffer && z) {
      const cudaError_t e2 = cudaFreeAsync(z, s);
      if (e == cudaSuccess) e = e2;
    }
    return status_of(e);
  }
  char* base = static_cast<char*>(dev_buffer);
  cudaError_t e = cudaSuccess;
  if (!base) e = cudaMallocAsync(reinterpret_cast<void**>(&base), need, s);
  if (e != cudaSuccess) return RET_ERR_CUDA;

  {
    std::lock_guard<std::mutex> hold(g_pipe_lock[dev]);
    Pipe* P = nullptr;
    e = pipe_for(dev, &P);
    if (e == cudaSuccess) e = cudaEventRecord(P->fork, s);
    bool forked[kSlots] = {};
    const char* hq = static_cast<const char*>(q);
    const char* hk = static_cast<const char*>(k);
    const char* hv = static_cast<const char*>(v);
    char* ho = static_cast<char*>(out);
    char* hs = reinterpret_cast<char*>(state_out);
    for (int i = 0; i < sl.count && e == cudaSuccess; ++i) {
      const int slot = i % kSlots;
      cudaStream_t ss = P->st[slot];
      if (!forked[slot]) {
        e = cudaStreamWaitEvent(ss, P->fork, 0);
        if (e != cudaSuccess) break;
        forked[slot] = true;
      }
      const SlabShape sh = slab_shape(sl, B, H, i);
      const size_t pairs = (size_t)sh.B * sh.H, rows = pairs * N;
      char* d = base + (size_t)slot * L.bytes;
      const size_t nq = rows * dk * 2, nv = rows * dv * 2;
      const size_t r0 = (size_t)sh.bh0 * N;
      e = cudaMemcpyAsync(d + L.q, hq + r0 * dk * 2, nq, cudaMemcpyHostToDevice, ss);
      if (e == cudaSuccess) e = cudaMemcpyAsync(d + L.k, hk + r0 * dk * 2, nq, cudaMemcpyHostToDevice, ss);
      if (e == cudaSuccess) e = cudaMemcpyAsync(d + L.v, hv + r0 * dv * 2, nv, cudaMemcpyHostToDevice, ss);
      ret::ChunkPlan plan;
      if (e == cudaSuccess && !ret::chunk_tc_plan(sh.B, sh.H, N, dk, dv, chunk, sms, &plan, L.ws_bytes))
        e = cudaErrorNotSupported;
      // a slab of one batch row's heads reads its heads' decays from gamma + bh0
      const float* g = sl.whole_rows ? gamma : gamma + sh.bh0;
      if (e == cudaSuccess)
        e = ret::launch_chunk_tc(d + L.q, d + L.k, d + L.v, g, nullptr, d + L.o,
                                 state_out ? reinterpret_cast<float*>(d + L.st) : nullptr, sh.B, sh.H, N, dk, dv, plan,
                                 plan.workspace_bytes ? reinterpret_cast<float*>(d + L.ws) : nullptr, nullptr, 0.f, ss);
      if (e == cudaSuccess) e = cudaMemcpyAsync(ho + r0 * dv * 2, d + L.o, nv, cudaMemcpyDeviceToHost, ss);
      if (e == cudaSuccess && state_out)
        e = cudaMemcpyAsync(hs + (size_t)sh.bh0 * st_row, d + L.st, pairs * st_row, cudaMemcpyDeviceToHost, ss);
    }
    // join whatever was forked, whether or not every step went in
    for (int j = 0; j < kSlots; ++j) {
      if (!forked[j]) continue;
      cudaError_t ej = cudaEventRecord(P->join[j], P->st[j]);
      if (ej == cudaSuccess) ej = cudaStreamWaitEvent(s, P->join[j], 0);
      if (e == cudaSuccess) e = ej;
    }
  }
  if (!dev_buffer) {
    const cudaError_t e2 = cudaFreeAsync(base, s);
    if (e == cudaSuccess) e = e2;
  }
  if (e == cudaErrorNotSupported) return RET_ERR_UNSUPPORTED;
  return status_of(e);
}

}  // extern "C"
