// internal.h -- declarations shared by the library's translation units.
// Not part of the public ABI (that is include/retention.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstddef>
#include <cstdint>

namespace ret {

// Largest dynamic shared memory a block may opt into on sm_100-class parts.
constexpr int kMaxSmemPerBlock = 232448;  // 227 KB

// ---- SIMT kernels (simt.cu) -------------------------------------------------
// Each returns a cudaError_t from the launch (cudaGetLastError after it).
// theta (nullable): q and k are first turned by the position phase rotation
// of the token at position pos.
cudaError_t launch_step_bf16(const void* q, const void* k, const void* v, float* state, void* out,
                             int B, int H, int dk, int dv, cudaStream_t s, const float* theta = nullptr,
                             int pos = 0);
cudaError_t launch_step_f32(const float* q, const float* k, const float* v, float* state,
                            float* out, int B, int H, int dk, int dv, cudaStream_t s);
cudaError_t launch_parallel_bf16(const void* q, const void* k, const void* v, const float* gamma,
                                 void* out, int B, int H, int N, int dk, int dv, cudaStream_t s);
cudaError_t launch_parallel_f32(const float* q, const float* k, const float* v,
                                const float* gamma, float* out, int B, int H, int N, int dk,
                                int dv, cudaStream_t s);
// Shared memory bytes the fp32 chunkwise kernel needs (0 if dims are invalid).
size_t chunkwise_f32_smem_bytes(int dk, int chunk);
cudaError_t launch_chunkwise_f32(const float* q, const float* k, const float* v,
                                 const float* gamma, float* out, float* state_out, int B, int H,
                                 int N, int dk, int dv, int chunk, cudaStream_t s);

// ---- tensor-core chunkwise (chunk_tc.cu) --------------------------------------
// Tensor map of a [BH][N][d] bf16 tensor as 3-D (d, N, BH) with boxes of 64
// columns x `rows` rows and 128-byte swizzle; boxes past the ends read zeros.
// ld: elements between rows (0: d, the rows are packed); the map covers the
// first d columns of each row.
bool make_map(CUtensorMap* m, const void* base, int d, int N, int BH, int rows, int ld = 0);
struct ChunkPlan {
  int chunk;        // tokens per tile (64 or 128, whatever chunk was asked for)
  int dk_tile;      // query/key columns the kernel is built for (128 or 256; dk <= dk_tile)
  int dvt;          // value columns per CTA (64 or 128)
  int n_dv_tiles;   // ceil(dv / dvt); the last tile's columns past dv are padding
  int segments;     // sequence segments of each cut unit (>= 1; 1: nothing is cut)
  int seg_chunks;   // chunks per segment (all segments but the last are full)
  int full_units;   // units ((b*H+h) * n_dv_tiles + value tile) run whole; the rest are cut
  int n_chunks;     // ceil(N / chunk)
  size_t workspace_bytes;  // float32 segment states of the cut units, 0 if segments == 1
  int launches;     // kernels enqueued by one call
};
// Fills `plan` for a supported shape; returns false for unsupported shapes.
// When there are more units than SMs, the units of the last, partial wave are
// cut into segments only if their segment states take at most ws_limit bytes
// (otherwise every unit runs whole and no workspace is needed).
// tile: 0 lets the plan pick the tile height (64 or 128 tokens, see
// chunk_tc.cu), 64 or 128 fixes it.
bool chunk_tc_plan(int B, int H, int N, int dk, int dv, int chunk, int num_sms, ChunkPlan* plan,
                   size_t ws_limit = SIZE_MAX, int tile = 0);
// Workspace bytes of the plan that retention_chunkwise_ws runs when given at
// most `limit` bytes (a RET_* status; plans on the current device).
int chunkwise_workspace_within(int B, int H, int N, int dk, int dv, int chunk, size_t limit, size_t* bytes);
// Kernels a call with this plan enqueues (2 when the sequence is split:
// state-only pre-pass, then main pass).
int chunk_tc_launch_count(const ChunkPlan& plan);
// GroupNorm of the outputs fused into the chunkwise epilogue (one value tile
// per head): weight, bias [H dv] (nullable: one, zero) and eps; the outputs are
// then written [B][N][H][dv].
struct ChunkNorm {
  const float* weight;
  const float* bias;
  float eps;
};
// Position phase rotation applied to q and k inside the kernel: frequencies
// theta [dk/2] (device), position of token 0.
struct ChunkRotation {
  const float* theta;
  int n0;
};
// state_in (nullable) is the state before the first token, [B*H][dk][dv];
// norm (nullable) selects the GroupNorm epilogue; scale multiplies the query
// (<= 0: 1/sqrt(dk)); rot (nullable) turns q and k by their positions first.
// ldqk: elements between the rows of q and of k (0: dk; a larger value reads
// dk columns of wider rows).  rev runs time backwards: out_m = scale sum_{n>=m} gamma^(n-m) (q_m . k_n) v_n
// + scale gamma^(N-m) q_m state_in, state_out = gamma^N state_in + sum_n
// gamma^n k_n^T v_n (not with norm or rot).
cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* gamma,
                            const float* state_in, void* out, float* state_out, int B, int H,
                            int N, int dk, int dv, const ChunkPlan& plan, float* workspace,
                            const ChunkNorm* norm, float scale, cudaStream_t s,
                            const ChunkRotation* rot = nullptr, bool rev = false, int ldqk = 0);
cudaError_t read_device_status(unsigned int* flags, int clear);
// Failure-path test setting read by every chunkwise launch (0: off).
extern std::atomic<unsigned int> g_test_stall_us;

// ---- gradients of the forward on the CUDA cores (backward.cu) ------------------
// The chunk length the kernel uses inside and its dynamic shared memory for
// these widths.
int backward_chunk(int dk, int dv);
size_t backward_smem_bytes(int dk, int dv);
cudaError_t launch_backward(bool bf16, const void* q, const void* k, const void* v, const float* gamma,
                            const float* state_in, const void* dout, const float* dstate, void* dq, void* dk_out,
                            void* dv_out, float* dstate_in, int B, int H, int N, int dk, int dv, cudaStream_t s);

// ---- parallel form on the tensor cores (parallel_tc.cu) ------------------------
bool parallel_tc_supported(int dk, int dv);
cudaError_t launch_parallel_tc(const void* q, const void* k, const void* v, const float* gamma, void* out, int B,
                               int H, int N, int dk, int dv, cudaStream_t s);
// Reads (and with `clear`, zeroes) the parallel kernels' device status word.
cudaError_t read_parallel_status(unsigned int* flags, int clear);

// ---- gradients of the forward on the tensor cores (bwd_tc.cu) -----------------
// Widths the tensor-core gradients handle (each gradient is a chunkwise
// forward of permuted operands, so both widths must be forward widths).
bool backward_tc_supported(int dk, int dv);
cudaError_t launch_backward_tc(const void* q, const void* k, const void* v, const float* gamma, const float* state_in,
                               const void* dout, const float* dstate, void* dq, void* dk_out, void* dv_out,
                               float* dstate_in, int B, int H, int N, int dk, int dv, cudaStream_t s);
// Kernels one such call enqueues on a GPU with 148 SMs (-1: unsupported).
int backward_tc_launches(int B, int H, int N, int dk, int dv, bool has_state_in, bool has_dstate, bool want_dstate_in);

// ---- position phase rotation of queries and keys (rotate.cu) -------------------
bool rotate_supported(int N, int d, int n0);
cudaError_t launch_rotate_bf16(const void* x, const float* theta, void* y, int B, int H, int N, int d,
                               int n0, cudaStream_t s);

// ---- normalisation of the heads' outputs (groupnorm.cu) -----------------------
bool groupnorm_supported(int dv);
cudaError_t launch_groupnorm_bf16(const void* r, const float* weight, const float* bias, void* y, int B,
                                  int H, int N, int dv, float eps, cudaStream_t s);

}  // namespace ret
