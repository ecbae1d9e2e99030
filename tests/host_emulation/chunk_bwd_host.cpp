// Host run of the backward's block bodies (chunked_recurrence_gb300/csrc/chunk_bwd_body.cuh),
// for the CPU tests: the same code the CUDA kernels run, kernel after kernel, with every
// block and every parallel item executed in order by one thread.  fp32 inputs only.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "chunk_bwd_body.cuh"

namespace {

struct HostExec {
  template <class F>
  void par(int n, F &&f) {
    for (int i = 0; i < n; ++i) f(i);
  }
  void sync() {}
  bool leader() const { return true; }
  void add(float *p, float v) { *p += v; }
  void fail(int32_t *status) {
    if (status && *status == 0) *status = 6;  // GDN_ERR_BOUNDS
  }
};

struct HostLoad {
  static constexpr bool kRawTf32 = false;
  float operator()(const void *p, int64_t i) const { return reinterpret_cast<const float *>(p)[i]; }
  void vec8(const void *p, int64_t i, float *out) const {
    for (int e = 0; e < 8; ++e) out[e] = reinterpret_cast<const float *>(p)[i + e];
  }
};

}  // namespace

template <int K>
void run_all(gdn_bwd::Params &p, int n_seqs, int64_t n_slots) {
  HostExec x;
  std::vector<float> sm(std::max(gdn_bwd::prep_smem_floats(K),
                                 std::max(gdn_bwd::walk_smem_floats(K, 32), gdn_bwd::grad_smem_floats(K))));
  for (int64_t slot = 0; slot < n_slots; ++slot)
    for (int h = 0; h < p.Hv; ++h) gdn_bwd::prep_block<K>(x, p, HostLoad{}, sm.data(), slot, h);
  const int bv = p.V % 32 == 0 ? 32 : 16;
  for (int s = 0; s < n_seqs; ++s)
    for (int h = 0; h < p.Hv; ++h)
      for (int tile = 0; tile < p.V / bv; ++tile) {
        if (bv == 32) gdn_bwd::walk_block<K, 32>(x, p, HostLoad{}, sm.data(), tile, h, s);
        else gdn_bwd::walk_block<K, 16>(x, p, HostLoad{}, sm.data(), tile, h, s);
      }
  for (int64_t slot = 0; slot < n_slots; ++slot)
    for (int h = 0; h < p.Hv; ++h) gdn_bwd::grad_block<K>(x, p, HostLoad{}, sm.data(), slot, h);
}

// -1: vector loads where the shapes allow them (as the library decides for aligned inputs);
// 0: the element-wise loads the library takes for unaligned inputs
static int g_vec8 = -1;
extern "C" void emu_set_vec8(int mode) { g_vec8 = mode; }

extern "C" int emu_chunk_bwd(const float *q, const float *k, const float *v, const float *g, const float *beta,
                             const float *h0, const int32_t *cu, int n_seqs, int64_t row_T, int64_t n_tok, int Hqk,
                             int Hv, int K, int V, float scale, int l2norm, const float *dout, const float *dhT,
                             float *dq, float *dk, float *dv, float *dg, float *dbeta, float *dh0) {
  const int64_t n_slots = n_seqs + (n_tok + gdn_bwd::C - 1) / gdn_bwd::C;
  std::vector<float> states((size_t)n_slots * Hv * V * K), dqn((size_t)n_tok * Hqk * K), dkn(dqn.size());
  std::vector<float> prep((size_t)n_slots * Hv * gdn_bwd::kPrep), sums((size_t)n_slots * Hv * gdn_bwd::kSums);
  std::vector<float> fw((size_t)n_slots * Hv * 3 * gdn_bwd::C * V);
  if (n_tok > 0) {
    std::memset(dv, 0, sizeof(float) * (size_t)n_tok * Hv * V);
    std::memset(dg, 0, sizeof(float) * (size_t)n_tok * Hv);
    std::memset(dbeta, 0, sizeof(float) * (size_t)n_tok * Hv);
  }
  int32_t status = 0;
  gdn_bwd::Params p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.h0 = h0; p.dout = dout; p.dhT = dhT;
  p.cu = cu; p.row_T = row_T; p.n_tok = n_tok; p.n_seqs = n_seqs;
  p.Hqk = Hqk; p.Hv = Hv; p.K = K; p.V = V;
  p.qs = (int64_t)Hqk * K; p.ks = (int64_t)Hqk * K; p.vs = (int64_t)Hv * V;
  p.scale = scale; p.l2norm = l2norm;
  p.vec8 = (g_vec8 != 0 && K % 8 == 0 && V % 8 == 0) ? 1 : 0;
  p.states = states.data(); p.fw = fw.data(); p.prep = prep.data(); p.sums = sums.data();
  p.dqn = dqn.data(); p.dkn = dkn.data();
  p.dv = dv; p.dg = dg; p.dbeta = dbeta; p.dh0 = dh0; p.status = &status;
  if (K == 32) run_all<32>(p, n_seqs, n_slots);
  else if (K == 64) run_all<64>(p, n_seqs, n_slots);
  else run_all<128>(p, n_seqs, n_slots);
  for (int64_t r = 0; r < n_tok * Hqk; ++r) {
    gdn_bwd::l2_back_row(q, p.qs, Hqk, K, l2norm, HostLoad{}, dqn.data(), dq, r);
    gdn_bwd::l2_back_row(k, p.ks, Hqk, K, l2norm, HostLoad{}, dkn.data(), dk, r);
  }
  return status;
}
