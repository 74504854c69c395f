// Tensor-core (tcgen05) weight-streaming GEMM: plans and launcher.
#pragma once

#include <memory>
#include <string>
#include <vector>

#include "internal.h"

namespace wedlm {

struct TcMapTable;  // TMA descriptors of every weight matrix

// Everything the bf16 GEMMs need that is fixed at create time.
struct TcPlanSet {
  int num_sms = 0;
  size_t part_elems = 0;
  std::shared_ptr<TcMapTable> maps;
};

int tc_choose_splits(int tiles, int nkb, int M, int N, int ntile, int num_sms,
                     size_t part_elems, double* time_out = nullptr);

std::unique_ptr<TcPlanSet> make_tc_plans(const wedlm_config& g,
                                         const std::vector<LayerWeights>& layers,
                                         const void* embed, const void* lm_head,
                                         void* xn, void* o, void* act,
                                         int num_sms, size_t part_elems,
                                         std::string* msg);

struct TcChoice {
  int ntile;     // output features per tile
  int splits;    // K splits
};
// *t_out (may be null): the modelled time of the plan, seconds
TcChoice tc_plan(const TcPlanSet& plans, const GemmProblem& P, double* t_out = nullptr);

// Launches one GEMM; *tiles_out (may be null) receives the number of
// output-feature tiles (the LM head's softmax records per row) and
// *launches_out (may be null) the number of kernels enqueued (2 with split-K).
cudaError_t launch_gemm_tc(const TcPlanSet& plans, GemmProblem P, int kind,
                           cudaStream_t st, int* tiles_out, int* launches_out);

}  // namespace wedlm
