// Single-launch f32 path for small TT layers (the 64 x 64, 16-token layer and
// its kin): one CTA runs the whole pass in shared memory with exact fp32
// fused multiply-adds, so a forward or a backward is one kernel launch with no
// intermediate in device memory.
//
// The contraction order is the one of the CoMERA project page ("Making small
// tensor operations fast on GPUs", bullet "One contraction order for both
// passes"): the input-side cores are merged into A (N x r_d) and the output-side
// cores into B (r_d x M), then z = x A, z' = z diag(D_d), y = z' B.  The
// backward runs the same path in reverse and takes the core and diagonal
// gradients through the merges with the left prefixes P_k:
//   P_k[(u, s), b] = sum_a P_{k-1}[u, a] D[a] G[a, s, b]
//   dG[a, s, b]    = D[a] sum_u P_{k-1}[u, a] dP_k[(u, s), b]
//   dQ[u, a]       = sum_{s, b} dP_k[(u, s), b] G[a, s, b]
//   dD[a]          = sum_u P_{k-1}[u, a] dQ[u, a]      (0 where D[a] == 0)
//   dP_{k-1}[u, a] = D[a] dQ[u, a]
#include <cuda_runtime.h>

#include "tc_fused.h"
#include "ttc_internal.h"

namespace ttc {
namespace {

constexpr int kSmallThreads = 512;
constexpr int kSmallMaxFloats = 50 * 1024;  // 200 KB of shared memory

struct SmallArgs {
  int d, K;
  int s[kMaxK];
  int r[kMaxK + 1];
  int U[kMaxK];             // rows of the prefix product ending at core k
  int core_off[kMaxK];
  int diag_off[kMaxK - 1];
  int n_floats;
  int T, N, M, rd;
  int acc;                  // backward: add into dparams
  // shared-memory offsets (floats)
  int o_prm, o_P[kMaxK], o_x, o_g, o_z, o_dz, o_dP0, o_dP1;
  const float* x;           // forward: x; backward: x
  const float* dy;
  const float* params;
  float* out;               // forward: y; backward: dx
  float* dparams;
  float* pout[kMaxK];       // forward: where to leave the prefix products (null: nowhere)
};

// C[m][n] (=|+=) sum_k A[m][k] B[k][n] with element (i, j) of X at
// X[i * si + j * sj] (shared or global addresses alike); one thread per output.
__device__ void sgemm(int m, int n, int kk, const float* A, int sam, int sak, const float* B,
                      int sbk, int sbn, float* C, int scm, int scn, bool acc) {
  for (int o = threadIdx.x; o < m * n; o += blockDim.x) {
    const int i = o / n, j = o - (o / n) * n;
    float v = 0.f;
    for (int k = 0; k < kk; ++k) v = fmaf(A[i * sam + k * sak], B[k * sbk + j * sbn], v);
    float* c = C + i * scm + j * scn;
    *c = acc ? *c + v : v;
  }
}

// Prefix products of one side, cores k0 .. k1 (P_{k0} is the first core).
__device__ void merge_side(const SmallArgs& a, float* sm, int k0, int k1) {
  const float* prm = sm + a.o_prm;
  float* P0 = sm + a.o_P[k0];
  const int n0 = a.U[k0] * a.r[k0 + 1];
  for (int i = threadIdx.x; i < n0; i += blockDim.x) P0[i] = prm[a.core_off[k0] + i];
  __syncthreads();
  for (int k = k0 + 1; k <= k1; ++k) {
    // P_k[(u, s), b] = sum_a P_{k-1}[u, a] D_{k-1}[a] G_k[a, s, b]
    const float* Pp = sm + a.o_P[k - 1];
    const float* D = prm + a.diag_off[k - 1];
    const float* G = prm + a.core_off[k];
    float* P = sm + a.o_P[k];
    const int ra = a.r[k], sk = a.s[k], rb = a.r[k + 1], U = a.U[k - 1];
    for (int o = threadIdx.x; o < U * sk * rb; o += blockDim.x) {
      const int u = o / (sk * rb), sb = o - u * (sk * rb);
      float v = 0.f;
      for (int x = 0; x < ra; ++x) v = fmaf(Pp[u * ra + x] * D[x], G[x * sk * rb + sb], v);
      P[o] = v;
    }
    __syncthreads();
  }
}

__device__ void merge_all(const SmallArgs& a, float* sm) {
  float* prm = sm + a.o_prm;
  for (int i = threadIdx.x; i < a.n_floats; i += blockDim.x) prm[i] = a.params[i];
  __syncthreads();
  merge_side(a, sm, 0, a.d - 1);
  merge_side(a, sm, a.d, a.K - 1);
}

__global__ void __launch_bounds__(kSmallThreads) small_fwd_kernel(SmallArgs a) {
  extern __shared__ float sm[];
  merge_all(a, sm);
  // the prefix products for a later backward that reuses this forward's merge
  for (int k = 0; k < a.K; ++k) {
    if (!a.pout[k]) continue;
    const float* P = sm + a.o_P[k];
    for (int i = threadIdx.x; i < a.U[k] * a.r[k + 1]; i += blockDim.x) a.pout[k][i] = P[i];
  }
  const float* A = sm + a.o_P[a.d - 1];   // N x rd
  const float* B = sm + a.o_P[a.K - 1];   // rd x M
  const float* Dd = sm + a.o_prm + a.diag_off[a.d - 1];
  float* z = sm + a.o_z;
  // z' = (x A) diag(D_d), x read straight from global memory
  for (int o = threadIdx.x; o < a.T * a.rd; o += blockDim.x) {
    const int t = o / a.rd, c = o - t * a.rd;
    float v = 0.f;
    for (int j = 0; j < a.N; ++j) v = fmaf(a.x[(size_t)t * a.N + j], A[j * a.rd + c], v);
    z[o] = v * Dd[c];
  }
  __syncthreads();
  sgemm(a.T, a.M, a.rd, z, a.rd, 1, B, a.M, 1, a.out, a.M, 1, false);
}

// Reverse steps of one side: dP of the side's last core is in sm + o_dP0.
// Writes dG of every core of the side and dD of every link inside it.
__device__ void reverse_side(const SmallArgs& a, float* sm, int k0, int k1) {
  const float* prm = sm + a.o_prm;
  float* dP = sm + a.o_dP0;
  float* dQ = sm + a.o_dP1;
  for (int k = k1; k > k0; --k) {
    const float* Pp = sm + a.o_P[k - 1];
    const float* D = prm + a.diag_off[k - 1];
    const float* G = prm + a.core_off[k];
    const int ra = a.r[k], sk = a.s[k], rb = a.r[k + 1], U = a.U[k - 1];
    float* dG = a.dparams + a.core_off[k];
    // dG_k[x, s, b] = D[x] sum_u P_{k-1}[u, x] dP[(u, s), b]
    for (int o = threadIdx.x; o < ra * sk * rb; o += blockDim.x) {
      const int x = o / (sk * rb), sb = o - x * (sk * rb);
      float v = 0.f;
      for (int u = 0; u < U; ++u) v = fmaf(Pp[u * ra + x], dP[u * sk * rb + sb], v);
      v *= D[x];
      dG[o] = a.acc ? dG[o] + v : v;
    }
    // dQ[u, x] = sum_{s, b} dP[(u, s), b] G[x, s, b]
    for (int o = threadIdx.x; o < U * ra; o += blockDim.x) {
      const int u = o / ra, x = o - u * ra;
      float v = 0.f;
      for (int sb = 0; sb < sk * rb; ++sb) v = fmaf(dP[u * sk * rb + sb], G[x * sk * rb + sb], v);
      dQ[o] = v;
    }
    __syncthreads();
    // dD_{k-1}[x] = sum_u P_{k-1}[u, x] dQ[u, x] (0 where D[x] == 0);
    // dP_{k-1}[u, x] = D[x] dQ[u, x]
    float* dD = a.dparams + a.diag_off[k - 1];
    for (int x = threadIdx.x; x < ra; x += blockDim.x) {
      float v = 0.f;
      for (int u = 0; u < U; ++u) v = fmaf(Pp[u * ra + x], dQ[u * ra + x], v);
      if (D[x] == 0.f) v = 0.f;
      if (a.acc) {
        if (D[x] != 0.f) dD[x] += v;
      } else {
        dD[x] = v;
      }
    }
    for (int o = threadIdx.x; o < U * ra; o += blockDim.x) dP[o] = D[o % ra] * dQ[o];
    __syncthreads();
  }
  // the first core of the side: dG = dP
  float* dG = a.dparams + a.core_off[k0];
  const int n0 = a.U[k0] * a.r[k0 + 1];
  for (int i = threadIdx.x; i < n0; i += blockDim.x) dG[i] = a.acc ? dG[i] + dP[i] : dP[i];
  __syncthreads();
}

__global__ void __launch_bounds__(kSmallThreads) small_bwd_kernel(SmallArgs a) {
  extern __shared__ float sm[];
  merge_all(a, sm);
  const float* A = sm + a.o_P[a.d - 1];   // N x rd
  const float* B = sm + a.o_P[a.K - 1];   // rd x M
  const float* Dd = sm + a.o_prm + a.diag_off[a.d - 1];
  float* x = sm + a.o_x;
  float* g = sm + a.o_g;                   // dy
  float* z = sm + a.o_z;                   // z (then unchanged)
  float* dz = sm + a.o_dz;                 // dz' (then dz)
  for (int i = threadIdx.x; i < a.T * a.N; i += blockDim.x) x[i] = a.x[i];
  for (int i = threadIdx.x; i < a.T * a.M; i += blockDim.x) g[i] = a.dy[i];
  __syncthreads();
  // z = x A ; dz' = dy B^T
  sgemm(a.T, a.rd, a.N, x, a.N, 1, A, a.rd, 1, z, a.rd, 1, false);
  sgemm(a.T, a.rd, a.M, g, a.M, 1, B, 1, a.M, dz, a.rd, 1, false);
  __syncthreads();
  // dD_d = sum_t z * dz' (0 where D_d == 0)
  float* dDd = a.dparams + a.diag_off[a.d - 1];
  for (int c = threadIdx.x; c < a.rd; c += blockDim.x) {
    float v = 0.f;
    for (int t = 0; t < a.T; ++t) v = fmaf(z[t * a.rd + c], dz[t * a.rd + c], v);
    if (Dd[c] == 0.f) v = 0.f;
    if (a.acc) {
      if (Dd[c] != 0.f) dDd[c] += v;
    } else {
      dDd[c] = v;
    }
  }
  __syncthreads();  // the column sums have read z and dz'
  // z' = z D_d, dz = dz' D_d (in place)
  for (int o = threadIdx.x; o < a.T * a.rd; o += blockDim.x) {
    const float dc = Dd[o % a.rd];
    z[o] *= dc;
    dz[o] *= dc;
  }
  __syncthreads();
  // dx = dz A^T (global), dA = x^T dz -> dP of the input side's last core,
  // dB = z'^T dy -> dP of the output side's last core (rows a_d, columns i)
  sgemm(a.T, a.N, a.rd, dz, a.rd, 1, A, 1, a.rd, a.out, a.N, 1, false);
  float* dP = sm + a.o_dP0;
  sgemm(a.N, a.rd, a.T, x, 1, a.N, dz, a.rd, 1, dP, a.rd, 1, false);
  __syncthreads();
  reverse_side(a, sm, 0, a.d - 1);
  sgemm(a.rd, a.M, a.T, z, 1, a.rd, g, a.M, 1, dP, a.M, 1, false);
  __syncthreads();
  reverse_side(a, sm, a.d, a.K - 1);
}

bool small_layout(const LayerPlan& L, int64_t T, SmallArgs* a) {
  if (L.act != TT_DT_F32 || T < 1 || T > 4096) return false;
  int64_t o = 0;
  auto take = [&](int64_t n) {
    const int64_t r = o;
    o += (n + 3) / 4 * 4;
    return (int)r;
  };
  a->o_prm = take((int64_t)L.n_floats);
  int64_t pmax = 0;
  for (int k = 0; k < L.K; ++k) {
    const int64_t n = L.U[k] * L.r[k + 1];
    a->o_P[k] = take(n);
    if (n > pmax) pmax = n;
  }
  a->o_dP0 = take(pmax);
  a->o_dP1 = take(pmax);
  a->o_x = take(T * L.N);
  a->o_g = take(T * L.M);
  a->o_z = take(T * L.rd);
  a->o_dz = take(T * L.rd);
  if (o > kSmallMaxFloats) return false;
  a->d = L.d;
  a->K = L.K;
  for (int k = 0; k < L.K; ++k) {
    a->s[k] = L.s[k];
    a->U[k] = (int)L.U[k];
    a->core_off[k] = (int)L.core_off[k];
  }
  for (int k = 0; k <= L.K; ++k) a->r[k] = L.r[k];
  for (int e = 0; e < L.K - 1; ++e) a->diag_off[e] = (int)L.diag_off[e];
  a->n_floats = (int)L.n_floats;
  a->T = (int)T;
  a->N = (int)L.N;
  a->M = (int)L.M;
  a->rd = L.rd;
  return true;
}

size_t small_smem_bytes(const SmallArgs& a) {
  return (size_t)(a.o_dz + (a.T * a.rd + 3) / 4 * 4) * sizeof(float);
}

cudaError_t set_small_attrs() {
  static PerDevice once;
  return once.get([] {
    cudaError_t e = cudaFuncSetAttribute(small_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmallMaxFloats * 4);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(small_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmallMaxFloats * 4);
    return e;
  });
}

}  // namespace

bool small_f32_supported(const LayerPlan& L, int64_t T) {
  SmallArgs a;
  return small_layout(L, T, &a);
}

tt_status small_f32_forward(const LayerPlan& L, int64_t T, const void* x, const float* params,
                            void* y, float* const* pout, cudaStream_t st) {
  SmallArgs a;
  if (!small_layout(L, T, &a)) return TT_ERR_UNSUPPORTED;
  if (set_small_attrs() != cudaSuccess) return TT_ERR_CUDA;
  for (int k = 0; k < kMaxK; ++k) a.pout[k] = (pout && k < L.K) ? pout[k] : nullptr;
  a.x = static_cast<const float*>(x);
  a.dy = nullptr;
  a.params = params;
  a.out = static_cast<float*>(y);
  a.dparams = nullptr;
  a.acc = 0;
  small_fwd_kernel<<<1, kSmallThreads, small_smem_bytes(a), st>>>(a);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

tt_status small_f32_backward(const LayerPlan& L, int64_t T, const void* x, const void* dy,
                             const float* params, void* dx, float* dparams, bool acc,
                             cudaStream_t st) {
  SmallArgs a;
  if (!small_layout(L, T, &a)) return TT_ERR_UNSUPPORTED;
  if (set_small_attrs() != cudaSuccess) return TT_ERR_CUDA;
  a.x = static_cast<const float*>(x);
  a.dy = static_cast<const float*>(dy);
  a.params = params;
  a.out = static_cast<float*>(dx);
  a.dparams = dparams;
  a.acc = acc ? 1 : 0;
  for (int k = 0; k < kMaxK; ++k) a.pout[k] = nullptr;
  small_bwd_kernel<<<1, kSmallThreads, small_smem_bytes(a), st>>>(a);
  count_launches(1);
  return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

}  // namespace ttc
