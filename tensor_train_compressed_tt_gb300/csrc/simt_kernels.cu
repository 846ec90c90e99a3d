// Plain SIMT (CUDA-core, fp32 FMA) kernels of libttc.
//
// These carry the f32-activation path (exact fp32 arithmetic, no tensor
// cores, so results stay within 1e-4 of the fp64 definition), the merges of
// the core chain and their backward (all T-independent and tiny), and the
// elementwise GELU of the FFN pair.
#include <cuda_bf16.h>

#include "ttc_internal.h"

namespace ttc {
namespace {

template <typename T>
__device__ __forceinline__ float ld_as_f32(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld_as_f32<float>(const float* p, int64_t i) {
  return p[i];
}
template <>
__device__ __forceinline__ float ld_as_f32<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st_from_f32(T* p, int64_t i, float v);
template <>
__device__ __forceinline__ void st_from_f32<float>(float* p, int64_t i, float v) {
  p[i] = v;
}
template <>
__device__ __forceinline__ void st_from_f32<__nv_bfloat16>(__nv_bfloat16* p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

template <typename T>
__device__ __forceinline__ float ld_c(const T* p, int64_t i) {
  return ld_as_f32<T>(p, i);
}

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

// 64x64 output tile per block, 4x4 per thread, K staged through shared
// memory 16 at a time.  gridDim.z splits K (only with kAtomic).
template <typename TA, typename TB, typename TC>
__global__ void __launch_bounds__(NT) gemm_kernel(GemmArgs g) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const TA* A = static_cast<const TA*>(g.A);
  const TB* B = static_cast<const TB*>(g.B);
  TC* C = static_cast<TC*>(g.C);
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
  int64_t kbeg = 0, kend = g.k;
  if (gridDim.z > 1) {
    int64_t chunk = (g.k + gridDim.z - 1) / gridDim.z;
    chunk = (chunk + BK - 1) / BK * BK;
    kbeg = (int64_t)blockIdx.z * chunk;
    kend = kbeg + chunk < g.k ? kbeg + chunk : g.k;
  }
  float acc[4][4] = {};
  for (int64_t k0 = kbeg; k0 < kend; k0 += BK) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int idx = tid + e * NT;  // 0..1023
      int mm = idx % BM, kk = idx / BM;
      int64_t gm = m0 + mm, gk = k0 + kk;
      float v = 0.f;
      if (gm < g.m && gk < kend) {
        v = ld_as_f32<TA>(A, gm * g.sam + gk * g.sak);
        if (g.kscale) v *= g.kscale[gk % g.klen];
      }
      As[kk][mm] = v;
      int nn = idx % BN;
      int64_t gn = n0 + nn;
      float w = 0.f;
      if (gn < g.n && gk < kend) w = ld_as_f32<TB>(B, gk * g.sbk + gn * g.sbn);
      Bs[kk][nn] = w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int64_t gm = m0 + ty * 4 + i;
    if (gm >= g.m) continue;
    float rs = g.rscale ? g.rscale[gm] : 1.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int64_t gn = n0 + tx * 4 + j;
      if (gn >= g.n) continue;
      float v = acc[i][j] * rs;
      if (g.cscale) v *= g.cscale[gn % g.clen];
      int64_t ci = gm * g.scm + gn * g.scn;
      if (g.mode == kAtomic) {
        atomicAdd(reinterpret_cast<float*>(C) + ci, v);
      } else if (g.mode == kAccumulate) {
        st_from_f32<TC>(C, ci, ld_c<TC>(C, ci) + v);
      } else {
        st_from_f32<TC>(C, ci, v);
      }
    }
  }
}

template <typename TA, typename TB, typename TC>
cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t st) {
  dim3 grid((unsigned)((g.n + BN - 1) / BN), (unsigned)((g.m + BM - 1) / BM), 1);
  if (g.mode == kAtomic) {
    // split K so that the grid covers the GPU a few times over
    int64_t tiles = (int64_t)grid.x * grid.y;
    int64_t want = (600 + tiles - 1) / tiles;
    int64_t maxs = (g.k + 4 * BK - 1) / (4 * BK);
    int64_t z = want < maxs ? want : maxs;
    if (z < 1) z = 1;
    if (z > 65535) z = 65535;
    grid.z = (unsigned)z;
  }
  gemm_kernel<TA, TB, TC><<<grid, NT, 0, st>>>(g);
  count_launches(1);
  return cudaGetLastError();
}

__global__ void coldot_kernel(int64_t nrows, int ncols, const float* X, int64_t sx,
                              const float* Y, int64_t sy, const float* mask, float* out,
                              int accumulate) {
  const int c = blockIdx.x;
  float s = 0.f;
  for (int64_t u = threadIdx.x; u < nrows; u += blockDim.x) s += X[u * sx + c] * Y[u * sy + c];
  __shared__ float red[32];
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    s = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) {
      bool keep = !mask || mask[c] != 0.f;
      if (accumulate) {
        if (keep) out[c] += s;
      } else {
        out[c] = keep ? s : 0.f;
      }
    }
  }
}

__global__ void scale_periodic_kernel(int64_t n, const float* in, const float* scale, int len,
                                      float* out, int accumulate) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v = in[i];
    if (scale) v *= scale[i % len];
    out[i] = accumulate ? out[i] + v : v;
  }
}

// The normal CDF Phi(h) = (1 + erf(h / sqrt 2)) / 2 with erf from
// Abramowitz and Stegun, Handbook of Mathematical Functions, formula 7.1.26:
//   erf(x) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2),
//   t = 1 / (1 + p x),  x >= 0,  |error| <= 1.5e-7,
// (odd in x).  exp(-x^2) = exp(-h^2 / 2) is also the density's exponential,
// so GELU' = Phi + h phi costs one exponential.  The error is about one ulp
// of fp32 at 1, far below the rounding of a bf16 result.
struct NormalParts {
  float Phi, phi;
};
__device__ __forceinline__ NormalParts normal_parts(float h) {
  const float x = fabsf(h) * 0.70710678118654752f;
  const float t = __frcp_rn(fmaf(0.3275911f, x, 1.f));
  float poly = fmaf(1.061405429f, t, -1.453152027f);
  poly = fmaf(poly, t, 1.421413741f);
  poly = fmaf(poly, t, -0.284496736f);
  poly = fmaf(poly, t, 0.254829592f);
  poly *= t;
  const float e = __expf(-x * x);           // exp(-h^2 / 2)
  const float q = 0.5f * poly * e;          // (1 - erf(x)) / 2 = Phi(-|h|)
  NormalParts r;
  r.Phi = h >= 0.f ? 1.f - q : q;
  r.phi = 0.39894228040143268f * e;         // exp(-h^2 / 2) / sqrt(2 pi)
  return r;
}
__device__ __forceinline__ float gelu_f(float h) { return h * normal_parts(h).Phi; }
__device__ __forceinline__ float gelu_grad_f(float h) {
  const NormalParts n = normal_parts(h);
  return fmaf(h, n.phi, n.Phi);
}

template <typename TO>
__global__ void gelu_fwd_kernel(int64_t n, const float* h, TO* a) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    st_from_f32<TO>(a, i, gelu_f(h[i]));
}

__global__ void gelu_bwd_kernel(int64_t n, const float* h, float* da) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    da[i] *= gelu_grad_f(h[i]);
}

// bf16 in / bf16 out, 8 elements (one 16-byte word) at a time; each thread
// issues the loads of kWords words before using any, so that enough bytes
// are in flight per SM to run at the HBM rate.
constexpr int kWords = 4;

__device__ __forceinline__ uint4 gelu8(uint4 u) {
  __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(p[k]);
    p[k] = __floats2bfloat162_rn(gelu_f(f.x), gelu_f(f.y));
  }
  return u;
}
__device__ __forceinline__ uint4 gelu_grad8(uint4 uh, uint4 ud) {
  const __nv_bfloat162* ph = reinterpret_cast<const __nv_bfloat162*>(&uh);
  __nv_bfloat162* pd = reinterpret_cast<__nv_bfloat162*>(&ud);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 fh = __bfloat1622float2(ph[k]);
    const float2 fd = __bfloat1622float2(pd[k]);
    pd[k] = __floats2bfloat162_rn(fd.x * gelu_grad_f(fh.x), fd.y * gelu_grad_f(fh.y));
  }
  return ud;
}

__global__ void gelu_fwd_bf16_kernel(int64_t n8, const uint4* __restrict__ h, uint4* a) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < n8;
       i0 += stride * kWords) {
    uint4 u[kWords];
#pragma unroll
    for (int w = 0; w < kWords; ++w)
      if (i0 + w * stride < n8) u[w] = h[i0 + w * stride];
#pragma unroll
    for (int w = 0; w < kWords; ++w)
      if (i0 + w * stride < n8) a[i0 + w * stride] = gelu8(u[w]);
  }
}

__global__ void gelu_bwd_bf16_kernel(int64_t n8, const uint4* __restrict__ h, uint4* da) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < n8;
       i0 += stride * kWords) {
    uint4 uh[kWords], ud[kWords];
#pragma unroll
    for (int w = 0; w < kWords; ++w)
      if (i0 + w * stride < n8) {
        uh[w] = h[i0 + w * stride];
        ud[w] = da[i0 + w * stride];
      }
#pragma unroll
    for (int w = 0; w < kWords; ++w)
      if (i0 + w * stride < n8) da[i0 + w * stride] = gelu_grad8(uh[w], ud[w]);
  }
}

template <typename T>
__global__ void sum_into_kernel(int64_t n, T* out, const T* p0, const T* p1, int nparts) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v = ld_as_f32<T>(out, i);
    v += ld_as_f32<T>(p0, i);
    if (nparts > 1) v += ld_as_f32<T>(p1, i);
    st_from_f32<T>(out, i, v);
  }
}

unsigned grid_for(int64_t n, int threads) {
  int64_t b = (n + threads - 1) / threads;
  if (b > 65535LL * 8) b = 65535LL * 8;
  if (b < 1) b = 1;
  return (unsigned)b;
}

}  // namespace

cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t st) {
  if (g.m <= 0 || g.n <= 0) return cudaSuccess;
  using bf = __nv_bfloat16;
  const int key = g.ta * 4 + g.tb * 2 + g.tc;
  switch (key) {
    case 0: return launch_gemm<float, float, float>(g, st);
    case 1: return launch_gemm<float, float, bf>(g, st);
    case 2: return launch_gemm<float, bf, float>(g, st);
    case 3: return launch_gemm<float, bf, bf>(g, st);
    case 4: return launch_gemm<bf, float, float>(g, st);
    case 5: return launch_gemm<bf, float, bf>(g, st);
    case 6: return launch_gemm<bf, bf, float>(g, st);
    default: return launch_gemm<bf, bf, bf>(g, st);
  }
}

cudaError_t coldot(int64_t nrows, int ncols, const float* X, int64_t sx, const float* Y,
                   int64_t sy, const float* mask, float* out, bool accumulate,
                   cudaStream_t st) {
  if (ncols <= 0) return cudaSuccess;
  coldot_kernel<<<ncols, 256, 0, st>>>(nrows, ncols, X, sx, Y, sy, mask, out, accumulate);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t scale_periodic(int64_t n, const float* in, const float* scale, int len, float* out,
                           bool accumulate, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  scale_periodic_kernel<<<grid_for(n, 256), 256, 0, st>>>(n, in, scale, len, out, accumulate);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t gelu_fwd(int64_t n, const float* h, void* a, int ta, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (ta == TT_DT_BF16)
    gelu_fwd_kernel<__nv_bfloat16>
        <<<grid_for(n, 256), 256, 0, st>>>(n, h, static_cast<__nv_bfloat16*>(a));
  else
    gelu_fwd_kernel<float><<<grid_for(n, 256), 256, 0, st>>>(n, h, static_cast<float*>(a));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t gelu_fwd_bf16(int64_t n, const void* h, void* a, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (n % 8) return cudaErrorInvalidValue;
  gelu_fwd_bf16_kernel<<<grid_for((n / 8 + kWords - 1) / kWords, 256), 256, 0, st>>>(
      n / 8, static_cast<const uint4*>(h), static_cast<uint4*>(a));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t gelu_bwd_bf16(int64_t n, const void* h, void* da, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (n % 8) return cudaErrorInvalidValue;
  gelu_bwd_bf16_kernel<<<grid_for((n / 8 + kWords - 1) / kWords, 256), 256, 0, st>>>(
      n / 8, static_cast<const uint4*>(h), static_cast<uint4*>(da));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t sum_into(int64_t n, void* out, const void* const* parts, int nparts, int type,
                     cudaStream_t st) {
  if (n <= 0 || nparts <= 0) return cudaSuccess;
  if (nparts > 2) return cudaErrorInvalidValue;
  const void* p1 = nparts > 1 ? parts[1] : parts[0];
  if (type == TT_DT_BF16)
    sum_into_kernel<__nv_bfloat16><<<grid_for(n, 256), 256, 0, st>>>(
        n, static_cast<__nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(parts[0]),
        static_cast<const __nv_bfloat16*>(p1), nparts);
  else
    sum_into_kernel<float><<<grid_for(n, 256), 256, 0, st>>>(
        n, static_cast<float*>(out), static_cast<const float*>(parts[0]),
        static_cast<const float*>(p1), nparts);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t gelu_bwd(int64_t n, const float* h, float* da, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  gelu_bwd_kernel<<<grid_for(n, 256), 256, 0, st>>>(n, h, da);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace ttc
