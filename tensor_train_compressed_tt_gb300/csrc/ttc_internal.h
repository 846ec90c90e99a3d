// Internal declarations shared by the libttc translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "ttc.h"

namespace ttc {

constexpr int kMaxK = 2 * TT_MAX_D;  // cores per layer

// One TT layer after validation.  Core k (0-based) has shape
// (r[k], s[k], r[k+1]); diagonal e (0-based) sits on the link between core e
// and core e+1 and has r[e+1] entries; the middle diagonal is e = d-1.
struct LayerPlan {
  int d = 0, K = 0;
  int s[kMaxK] = {};
  int r[kMaxK + 1] = {};
  int64_t N = 0, M = 0;
  int rd = 0;         // middle rank r_d
  int act = TT_DT_F32;
  unsigned flags = 0;
  size_t core_off[kMaxK] = {};
  size_t diag_off[kMaxK - 1] = {};
  size_t n_floats = 0;
  // chain: U[k] = number of rows of the merged prefix ending at core k
  // (input side: s_0..s_k; output side: r_d * s_d..s_k)
  int64_t U[kMaxK] = {};
};

}  // namespace ttc

namespace ttc {
// TT-matrix embedding table: cores F_k (r_{k-1}, m_k, n_k, r_k), diagonals
// D_1..D_{d-1}; a table of two cores runs as three with a unit third core.
struct TtmPlan {
  int d = 0;                      // 2 or 3
  int m[3] = {1, 1, 1}, n[3] = {1, 1, 1}, r[4] = {1, 1, 1, 1};
  int64_t V = 0, Dm = 0;          // rows (prod m), width (prod n)
  int64_t npair = 0;              // distinct (i_1, i_2) prefixes: m_1 m_2
  size_t core_off[3] = {}, diag_off[2] = {}, n_floats = 0;
  unsigned flags = 0;
};
size_t ttm_workspace_bytes(const TtmPlan& P, int64_t B);
}  // namespace ttc

struct tt_plan_s {
  int kind = 0;  // 0 = single layer, 1 = FFN pair, 2 = TT-matrix embedding, 3 = layers on one x
  int G = 1;     // layers of a kind-3 plan
  ttc::LayerPlan L[3];
  ttc::TtmPlan ttm;
};

namespace ttc {

// ---- per-device set-up ------------------------------------------------------
// Kernel attributes (the shared-memory opt-in, the carveout) and occupancy
// figures belong to one device; a process that drives several GPUs needs them
// once on each.  A PerDevice runs its set-up step once for every device it is
// used on, with that device current, and keeps the result.
constexpr int kMaxDevices = 64;
class PerDevice {
 public:
  template <typename F>
  cudaError_t get(F&& fn) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
      return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (!done_[dev]) {
      res_[dev] = fn();
      done_[dev] = true;
    }
    return res_[dev];
  }

 private:
  std::mutex mu_;
  bool done_[kMaxDevices] = {};
  cudaError_t res_[kMaxDevices] = {};
};
// Streaming multiprocessors of the current device (cached per device; 1 if
// the query fails).
int device_sms();

// ---- device status word (one per GPU, module-scope device variable) -------
struct DeviceStatus {
  unsigned code;    // 0 = ok, else a tt_status value
  unsigned detail;  // where it happened (kernel-specific)
};
// Copies the current device's status word to *out and zeroes it.
cudaError_t read_and_clear_device_status(DeviceStatus* out);
// The same for the embedding kernels' own word (ttm.cu).
cudaError_t read_and_clear_ttm_status(DeviceStatus* out);

// ---- rank-adaptive step (rank_update.cu) ------------------------------------
// One elementwise launch of the step over a layer's packed params / dparams.
struct RankStep;
cudaError_t rank_update_launch(const LayerPlan& L, float* params, float* dparams,
                               const RankStep& r, cudaStream_t st);
// The step's weights from tt_rank_opts (false for negative or non-finite ones).
bool rank_step_from(const tt_rank_opts* opts, RankStep* r);

// ---- measurement hooks (profile.cu) ---------------------------------------
enum Phase { kPhMerge = 0, kPhFwd = 1, kPhBwd = 2, kPhMergeBwd = 3, kPhElem = 4 };
void prof_begin(int phase, cudaStream_t st);
void prof_end(int phase, cudaStream_t st);
void count_launches(int n);

// ---- SIMT kernels (simt_kernels.cu) ----------------------------------------
enum GemmMode { kStore = 0, kAccumulate = 1, kAtomic = 2 };

// C[m,n] (op)= rscale[m] * cscale[n % clen] * sum_k A[m,k] kscale[k % klen] B[k,n]
// Element (i,j) of X lives at X[i*si + j*sj].  Types: 0 = f32, 1 = bf16.
struct GemmArgs {
  int64_t m = 0, n = 0, k = 0;
  const void* A = nullptr; int64_t sam = 0, sak = 0; int ta = 0;
  const void* B = nullptr; int64_t sbk = 0, sbn = 0; int tb = 0;
  void* C = nullptr; int64_t scm = 0, scn = 0; int tc = 0;
  const float* kscale = nullptr; int klen = 1;
  const float* rscale = nullptr;
  const float* cscale = nullptr; int clen = 1;
  int mode = kStore;
};
cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t st);

// out[c] (=|+=) sum_u X[u*sx + c] * Y[u*sy + c], c < ncols; out[c] = 0 (or
// left unchanged when accumulating) where mask[c] == 0.
cudaError_t coldot(int64_t nrows, int ncols, const float* X, int64_t sx, const float* Y,
                   int64_t sy, const float* mask, float* out, bool accumulate,
                   cudaStream_t st);

// out[i] (=|+=) in[i] * scale[i % len]  (scale may be null: plain copy)
cudaError_t scale_periodic(int64_t n, const float* in, const float* scale, int len, float* out,
                           bool accumulate, cudaStream_t st);

// a = GELU(h) (exact erf form), written as f32 or bf16
cudaError_t gelu_fwd(int64_t n, const float* h, void* a, int ta, cudaStream_t st);
// dh = da * GELU'(h), in place over da (f32)
cudaError_t gelu_bwd(int64_t n, const float* h, float* da, cudaStream_t st);
// out[i] = out[i] + parts[0][i] + ... + parts[nparts-1][i], summed in f32 in
// that order and rounded once to out's type (TT_DT_F32 or TT_DT_BF16)
cudaError_t sum_into(int64_t n, void* out, const void* const* parts, int nparts, int type,
                     cudaStream_t st);
// bf16 variants (n a multiple of 8, 16-byte aligned buffers)
cudaError_t gelu_fwd_bf16(int64_t n, const void* h, void* a, cudaStream_t st);
cudaError_t gelu_bwd_bf16(int64_t n, const void* h, void* da, cudaStream_t st);

}  // namespace ttc
