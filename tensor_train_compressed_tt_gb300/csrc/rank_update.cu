// tt_rank_update: the penalty sub-gradient or one proximal gradient step of
// the early-stage rank-adaptive objective, elementwise over one layer's
// packed parameters (cores first, then the diagonals).
#include <cuda_runtime.h>

#include <cmath>

#include "ttc.h"
#include "ttc_internal.h"

namespace ttc {
namespace {

// n_core floats of cores, then n_diag floats of diagonals.  Each step is
// one IEEE float operation rounded to nearest (the _rn intrinsics keep the
// compiler from fusing a multiply into an add).
__global__ void rank_update_kernel(float* __restrict__ params, float* __restrict__ dparams,
                                   int n_core, int n_total, float b2, float gamma, float lr,
                                   float thr) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_total; i += gridDim.x * blockDim.x) {
    const float p = params[i];
    const float g = dparams[i];
    if (i < n_core) {
      const float grad = __fadd_rn(g, __fmul_rn(b2, p));
      if (lr == 0.f) dparams[i] = grad;
      else params[i] = __fsub_rn(p, __fmul_rn(lr, grad));
    } else if (lr == 0.f) {
      const float s = p > 0.f ? gamma : (p < 0.f ? -gamma : 0.f);
      dparams[i] = __fadd_rn(g, s);
    } else {
      const float v = __fsub_rn(p, __fmul_rn(lr, g));
      params[i] = v > thr ? __fsub_rn(v, thr) : (v < -thr ? __fadd_rn(v, thr) : 0.f);
    }
  }
}

bool ok_weight(float v) { return std::isfinite(v) && v >= 0.f; }

}  // namespace
}  // namespace ttc

using namespace ttc;

extern "C" tt_status tt_rank_update(const tt_plan_t* plan, float* params, float* dparams,
                                    const tt_rank_opts* opts, void* stream) {
  if (!plan || !params || !dparams || !opts || plan->kind != 0) return TT_ERR_INVALID_ARG;
  if (!ok_weight(opts->gamma) || !ok_weight(opts->beta) || !ok_weight(opts->lr))
    return TT_ERR_INVALID_ARG;
  const LayerPlan& L = plan->L[0];
  const int n_core = (int)L.diag_off[0];
  const int n_total = (int)L.n_floats;
  if (n_total <= 0) return TT_OK;
  const float b2 = 2.0f * opts->beta;  // exact
  const float thr = opts->lr * opts->gamma;  // one float32 product, as the step defines
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return TT_ERR_CUDA;
  int grid = (n_total + 255) / 256;
  if (grid > 4 * sms) grid = 4 * sms;
  rank_update_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      params, dparams, n_core, n_total, b2, opts->gamma, opts->lr, thr);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}
