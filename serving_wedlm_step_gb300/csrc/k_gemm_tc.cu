// bf16 weight-streaming GEMM entry (first version: CUDA-core mainloop).
#include "gemm_tc.h"

namespace wedlm {

std::unique_ptr<TcPlanSet> make_tc_plans(const wedlm_config& g,
                                         const std::vector<LayerWeights>& layers,
                                         const void* embed, const void* lm_head,
                                         void* xn, void* o, void* act,
                                         int num_sms, size_t part_elems,
                                         std::string* msg) {
  (void)g; (void)layers; (void)embed; (void)lm_head; (void)xn; (void)o; (void)act;
  (void)msg;
  std::unique_ptr<TcPlanSet> p(new TcPlanSet());
  p->num_sms = num_sms;
  p->part_elems = part_elems;
  return p;
}

cudaError_t launch_gemm_tc(const TcPlanSet& plans, GemmProblem P, int kind,
                           cudaStream_t st) {
  (void)kind;
  const int tiles = P.swiglu ? P.N / 128 : (P.N + 127) / 128;
  int s = std::max(1, 2 * plans.num_sms / std::max(1, tiles));
  s = std::min(s, std::max(1, P.K / 64));
  while (s > 1 && (size_t)s * P.M * P.N > plans.part_elems) --s;
  P.splits = s;
  return launch_gemm_simt<bf16>(P, st);
}

}  // namespace wedlm
