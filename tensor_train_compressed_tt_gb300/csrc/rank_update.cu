// tt_rank_update: the penalty sub-gradient or one proximal gradient step of
// the early-stage rank-adaptive objective, elementwise over one layer's
// packed parameters (cores first, then the diagonals).
#include <cuda_runtime.h>

#include <cmath>

#include "ttc.h"
#include "rank_step.cuh"
#include "ttc_internal.h"

namespace ttc {
namespace {

// n_core floats of cores, then n_diag floats of diagonals.
__global__ void rank_update_kernel(float* __restrict__ params, float* __restrict__ dparams,
                                   int n_core, int n_total, RankStep r) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_total; i += gridDim.x * blockDim.x)
    rank_step_elem(params, dparams, i, i < n_core, r);
}

bool ok_weight(float v) { return std::isfinite(v) && v >= 0.f; }

}  // namespace
}  // namespace ttc

namespace ttc {

bool rank_step_from(const tt_rank_opts* opts, RankStep* r) {
  if (!opts || !ok_weight(opts->gamma) || !ok_weight(opts->beta) || !ok_weight(opts->lr))
    return false;
  r->b2 = 2.0f * opts->beta;  // exact
  r->gamma = opts->gamma;
  r->lr = opts->lr;
  r->thr = opts->lr * opts->gamma;  // one float32 product, as the step defines
  return true;
}

cudaError_t rank_update_launch(const LayerPlan& L, float* params, float* dparams,
                               const RankStep& r, cudaStream_t st) {
  const int n_core = (int)L.diag_off[0];
  const int n_total = (int)L.n_floats;
  if (n_total <= 0) return cudaSuccess;
  int grid = (n_total + 255) / 256;
  if (grid > 4 * device_sms()) grid = 4 * device_sms();
  rank_update_kernel<<<grid, 256, 0, st>>>(params, dparams, n_core, n_total, r);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace ttc

using namespace ttc;

extern "C" tt_status tt_rank_update(const tt_plan_t* plan, float* params, float* dparams,
                                    const tt_rank_opts* opts, void* stream) {
  if (!plan || !params || !dparams || !opts || plan->kind != 0) return TT_ERR_INVALID_ARG;
  RankStep r;
  if (!rank_step_from(opts, &r)) return TT_ERR_INVALID_ARG;
  return rank_update_launch(plan->L[0], params, dparams, r, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? TT_OK
             : TT_ERR_CUDA;
}
