// One element of the rank-adaptive step of the early-stage objective
// L + gamma S_hat(D) + beta ||G||^2 (CoMERA project page, "Learn the ranks
// while training"), shared by the standalone update kernel and the merge
// engine's last phase.  Every step is one IEEE float operation rounded to
// nearest (the _rn intrinsics keep the compiler from fusing a multiply into
// an add), so both give the same bits.
//   core entry, lr == 0:  g <- g + 2 beta p
//   core entry, lr > 0:   p <- p - lr (g + 2 beta p)
//   diagonal,   lr == 0:  g <- g + gamma sign(p)          (sign(0) = 0)
//   diagonal,   lr > 0:   p <- soft_threshold(p - lr g, lr gamma)
#pragma once

#include <cuda_runtime.h>

namespace ttc {

struct RankStep {
  float b2;     // 2 beta
  float gamma;
  float lr;
  float thr;    // lr * gamma, one float product
};

__device__ __forceinline__ void rank_step_elem(float* params, float* dparams, int i, bool core,
                                               const RankStep& r) {
  const float p = params[i];
  const float g = dparams[i];
  if (core) {
    const float grad = __fadd_rn(g, __fmul_rn(r.b2, p));
    if (r.lr == 0.f) dparams[i] = grad;
    else params[i] = __fsub_rn(p, __fmul_rn(r.lr, grad));
  } else if (r.lr == 0.f) {
    const float s = p > 0.f ? r.gamma : (p < 0.f ? -r.gamma : 0.f);
    dparams[i] = __fadd_rn(g, s);
  } else {
    const float v = __fsub_rn(p, __fmul_rn(r.lr, g));
    params[i] = v > r.thr ? __fsub_rn(v, r.thr) : (v < -r.thr ? __fadd_rn(v, r.thr) : 0.f);
  }
}

}  // namespace ttc
