// Steps the phases of backward_kernel (backward.cu) on the CPU, thread by
// thread: for each CTA, each phase runs for all 256 thread indices before the
// next phase starts, which is what the kernel's barriers guarantee on the
// GPU.  Shared memory is a heap buffer of exactly the kernel's dynamic size,
// filled with NaN, so an out-of-range index shows up under AddressSanitizer
// and a read of a slot no phase wrote shows up as a non-finite gradient.  The
// per-chunk regions (a rows, b rows, the transposed w slab and the scores)
// are filled with NaN again before every chunk's load phase, so a phase that
// reads a slot of the current chunk it did not write cannot pick up the
// previous chunk's value; the state slab and the power table carry over.
// This is test code: the library never runs its kernels on the CPU.
//
// Input file: int32 header {bf16, B, H, N, dk, dv, has_state_in, has_dstate},
// then float32 q, k, v, dout, gamma, [state_in], [dstate].  Output file:
// float32 dq, dk, dv (rounded to the kernel's element type), dstate_in.
#include "../../linear_attention_sequence_02_b300/csrc/backward.cu"

#include <cstdio>
#include <cstdlib>
#include <vector>

using namespace ret;

namespace {

template <int C, typename T>
void step_all(const BwdArgs& p, int BH) {
  const size_t nf = BwdSmem<C>::floats(p.wmax);
  float* smem = static_cast<float*>(aligned_alloc(16, ((nf * sizeof(float) + 15) / 16) * 16));
  for (int bx = 0; bx < BH; ++bx)
    for (int by = 0; by < 2 * p.slabs_k + p.slabs_v; ++by) {
      for (size_t i = 0; i < nf; ++i) smem[i] = __builtin_nanf("");
      const BwdRole r = bwd_role(p, bx, by);
      const BwdSmem<C> s(smem, p.wmax);
      for (int t = 0; t < kBwdThreads; ++t) bwd_init<C>(p, r, s, t);
      const int n_chunks = (p.N + C - 1) / C;
      const size_t per_chunk = (size_t)(s.St - s.As);  // As, Bs, WT and P, contiguous
      for (int it = 0; it < n_chunks; ++it) {
        const int s0 = (r.fwd ? it : n_chunks - 1 - it) * C;
        const int L = imin(C, p.N - s0);
        for (size_t i = 0; i < per_chunk; ++i) s.As[i] = __builtin_nanf("");
        for (int t = 0; t < kBwdThreads; ++t) bwd_load<C, T>(p, r, s, s0, L, t);
        for (int t = 0; t < kBwdThreads; ++t) bwd_scores<C>(r, s, L, t);
        for (int t = 0; t < kBwdThreads; ++t) bwd_rows<C, T>(p, r, s, s0, L, t);
        for (int t = 0; t < kBwdThreads; ++t) bwd_update<C>(r, s, L, t);
      }
      for (int t = 0; t < kBwdThreads; ++t) bwd_final<C>(p, r, s, t);
    }
  free(smem);
}

template <typename T>
std::vector<T> as_type(const std::vector<float>& x) {
  std::vector<T> y(x.size());
  for (size_t i = 0; i < x.size(); ++i) y[i] = static_cast<T>(x[i]);
  return y;
}

template <typename T>
int run(FILE* in, FILE* out, int B, int H, int N, int dk, int dv, bool has_s0, bool has_ds) {
  auto read = [&](size_t n, std::vector<float>& v) {
    v.resize(n);
    return n == 0 || fread(v.data(), sizeof(float), n, in) == n;
  };
  const size_t nq = (size_t)B * H * N * dk, nv = (size_t)B * H * N * dv, ns = (size_t)B * H * dk * dv;
  std::vector<float> q, k, v, dout, gamma, s0, ds;
  if (!read(nq, q) || !read(nq, k) || !read(nv, v) || !read(nv, dout) || !read(H, gamma) ||
      !read(has_s0 ? ns : 0, s0) || !read(has_ds ? ns : 0, ds))
    return 3;
  std::vector<T> qt = as_type<T>(q), kt = as_type<T>(k), vt = as_type<T>(v), dt = as_type<T>(dout);
  std::vector<T> gq(nq), gk(nq), gv(nv);
  std::vector<float> ds0(ns, 0.f);
  BwdArgs a;
  a.q = qt.data();
  a.k = kt.data();
  a.v = vt.data();
  a.dout = dt.data();
  a.gamma = gamma.data();
  a.state_in = has_s0 ? s0.data() : nullptr;
  a.dstate = has_ds ? ds.data() : nullptr;
  a.grad_q = gq.data();
  a.grad_k = gk.data();
  a.grad_v = gv.data();
  a.dstate_in = ds0.data();
  a.H = H;
  a.N = N;
  a.dk = dk;
  a.dv = dv;
  a.slabs_k = (dk + kBwdSlab - 1) / kBwdSlab;
  a.slabs_v = (dv + kBwdSlab - 1) / kBwdSlab;
  a.wmax = dk > dv ? dk : dv;
  step_all<kBwdChunk, T>(a, B * H);
  for (const auto* g : {&gq, &gk, &gv})
    for (const T& e : *g) {
      const float f = static_cast<float>(e);
      fwrite(&f, sizeof(float), 1, out);
    }
  fwrite(ds0.data(), sizeof(float), ns, out);
  return 0;
}

}  // namespace

int main(int argc, char** argv) {
  if (argc != 3) return 2;
  FILE* in = fopen(argv[1], "rb");
  FILE* out = fopen(argv[2], "wb");
  if (!in || !out) return 2;
  int h[8];
  if (fread(h, sizeof(int), 8, in) != 8) return 2;
  const int rc = h[0] ? run<__nv_bfloat16>(in, out, h[1], h[2], h[3], h[4], h[5], h[6] != 0, h[7] != 0)
                      : run<float>(in, out, h[1], h[2], h[3], h[4], h[5], h[6] != 0, h[7] != 0);
  fclose(in);
  fclose(out);
  return rc;
}
