// TT-matrix (TTM) embedding lookup and its backward.
//
// Follows the CoMERA project page, "Making small tensor operations fast on
// GPUs", bullet "Embedding lookup without repeated work": only the distinct
// rows of a batch are computed, every distinct (i_1, i_2) prefix is
// contracted once (F_1 D_1 F_2 for that prefix: the pair product), and the
// rows are assembled from the pair products and the last core.  A two-core
// table runs as a three-core one whose third core and second diagonal are a
// single 1.
//
// Forward:  count -> scan -> pair products -> distinct rows -> scatter.
// Backward: count -> scan (+ row chunks) -> fill (occurrence lists) -> pair
//           products -> chunk sums of dout -> per distinct row: dF_3 and the
//           pair-product gradients -> per pair: dF_1, dF_2, dD_1, dD_2.
// Sums over repeated indices and over rows sharing a prefix use atomics.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>

#include "ttc.h"
#include "ttc_internal.h"

namespace ttc {
namespace {

constexpr int kChunk = 32;          // occurrences of one row summed per backward unit
constexpr int kMaxSmemFloats = 40960;

__device__ DeviceStatus g_ttm_status;
__device__ float g_ttm_one[4] = {1.f, 1.f, 1.f, 1.f};  // unit third core / second diagonal
__device__ float g_ttm_sink[64];                        // their gradients (discarded)

__device__ void ttm_error(unsigned where) {
  if (atomicCAS(&g_ttm_status.code, 0u, (unsigned)TT_ERR_DEVICE) == 0u)
    atomicExch(&g_ttm_status.detail, where);
}

struct TtmArgs {
  int B, V, npair;
  int m1, m2, m3, n1, n2, n3, r1, r2;
  int nA, Dm;                       // n1 n2, n1 n2 n3
  const float* F1;
  const float* F2;
  const float* F3;
  const float* D1;
  const float* D2;
  // workspace (cnt, cursor, cnt_pair adjacent: zeroed together per call)
  int* cnt;       // [V] occurrences of each row
  int* cursor;    // [V] fill cursors
  int* cnt_pair;  // [npair] prefix used
  int* off;       // [V] exclusive prefix of cnt (occurrence-list offsets)
  int* upos;      // [V] distinct-row slot of each used row
  int* ulist;     // [ucap] row of each distinct slot
  int* uoff;      // [ucap] first backward unit of each distinct slot
  int* unit_u;    // [units cap] distinct slot of each backward unit
  int* pos_pair;  // [npair] slot of each used prefix
  int* plist;     // [pcap] prefix of each slot
  int* counts;    // [4]: distinct rows, distinct prefixes, backward units
  int* occ;       // [B] occurrence lists
  float* P;       // [pcap][nA][r2] pair products F_1 D_1 F_2 (without D_2)
  float* dP;      // [pcap][nA][r2] gradient w.r.t. P * D_2
  float* rows;    // [ucap][Dm] distinct rows (forward) / [units][Dm] chunk sums (backward)
};

__global__ void ttm_count_kernel(TtmArgs a, const int32_t* __restrict__ idx) {
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < a.B; b += gridDim.x * blockDim.x) {
    const int v = idx[b];
    if (v < 0 || v >= a.V) {
      ttm_error(1);
      continue;
    }
    atomicAdd(a.cnt + v, 1);
    a.cnt_pair[v / a.m3] = 1;
  }
}

// Inclusive scan of 1024 per-thread values held in s (one block of 1024).
__device__ void block_scan_1024(int* s, int t) {
  for (int o = 1; o < 1024; o <<= 1) {
    const int x = t >= o ? s[t - o] : 0;
    __syncthreads();
    s[t] += x;
    __syncthreads();
  }
}

// One block of 1024 threads: occurrence offsets, distinct-row slots, backward
// units, and prefix slots, each an exclusive prefix sum over a contiguous
// segment per thread.
__global__ void __launch_bounds__(1024) ttm_scan_kernel(TtmArgs a) {
  __shared__ int s1[1024], s2[1024], s3[1024];
  const int t = threadIdx.x;
  const int chunk = (a.V + 1023) / 1024;
  const int lo = min(t * chunk, a.V), hi = min(lo + chunk, a.V);
  int c = 0, f = 0, u = 0;
  for (int v = lo; v < hi; ++v) {
    const int x = a.cnt[v];
    c += x;
    f += x > 0;
    u += (x + kChunk - 1) / kChunk;
  }
  s1[t] = c;
  s2[t] = f;
  s3[t] = u;
  __syncthreads();
  block_scan_1024(s1, t);
  block_scan_1024(s2, t);
  block_scan_1024(s3, t);
  int ec = t ? s1[t - 1] : 0, ef = t ? s2[t - 1] : 0, eu = t ? s3[t - 1] : 0;
  for (int v = lo; v < hi; ++v) {
    const int x = a.cnt[v];
    a.off[v] = ec;
    ec += x;
    if (x > 0) {
      a.upos[v] = ef;
      a.ulist[ef] = v;
      a.uoff[ef] = eu;
      const int nch = (x + kChunk - 1) / kChunk;
      for (int k = 0; k < nch; ++k) a.unit_u[eu + k] = ef;
      eu += nch;
      ++ef;
    }
  }
  if (t == 1023) {
    a.counts[0] = s2[1023];
    a.counts[2] = s3[1023];
  }
  __syncthreads();
  const int pch = (a.npair + 1023) / 1024;
  const int plo = min(t * pch, a.npair), phi = min(plo + pch, a.npair);
  f = 0;
  for (int p = plo; p < phi; ++p) f += a.cnt_pair[p] != 0;
  s2[t] = f;
  __syncthreads();
  block_scan_1024(s2, t);
  ef = t ? s2[t - 1] : 0;
  for (int p = plo; p < phi; ++p) {
    if (a.cnt_pair[p]) {
      a.pos_pair[p] = ef;
      a.plist[ef++] = p;
    }
  }
  if (t == 1023) a.counts[1] = s2[1023];
}

__global__ void ttm_fill_kernel(TtmArgs a, const int32_t* __restrict__ idx) {
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < a.B; b += gridDim.x * blockDim.x) {
    const int v = idx[b];
    if (v < 0 || v >= a.V) continue;
    a.occ[a.off[v] + atomicAdd(a.cursor + v, 1)] = b;
  }
}

// Pair products P[c][(j1, j2), e] = sum_b F_1[0, i1, j1, b] D_1[b] F_2[b, i2, j2, e]
// for every used prefix p = i1 m2 + i2 (slot c); with zero_dp also dP[c] = 0.
__global__ void ttm_pairs_kernel(TtmArgs a, int zero_dp) {
  extern __shared__ float sm[];
  const int n1 = a.n1, n2 = a.n2, r1 = a.r1, r2 = a.r2;
  float* f1 = sm;             // [n1][r1], times D_1
  float* f2 = f1 + n1 * r1;   // [r1][n2][r2]
  const int Pn = a.counts[1];
  const int nt = a.nA * r2;
  for (int c = blockIdx.x; c < Pn; c += gridDim.x) {
    const int p = a.plist[c];
    const int i1 = p / a.m2, i2 = p - (p / a.m2) * a.m2;
    for (int e = threadIdx.x; e < n1 * r1; e += blockDim.x)
      f1[e] = a.F1[i1 * n1 * r1 + e] * a.D1[e % r1];
    const int w2 = n2 * r2;
    for (int e = threadIdx.x; e < r1 * w2; e += blockDim.x) {
      const int b = e / w2;
      f2[e] = a.F2[(b * a.m2 + i2) * w2 + (e - b * w2)];
    }
    __syncthreads();
    float* out = a.P + (size_t)c * nt;
    for (int o = threadIdx.x; o < nt; o += blockDim.x) {
      const int jA = o / r2, e = o - (o / r2) * r2;
      const int j1 = jA / n2, j2 = jA - (jA / n2) * n2;
      float acc = 0.f;
      for (int b = 0; b < r1; ++b) acc = fmaf(f1[j1 * r1 + b], f2[(b * n2 + j2) * r2 + e], acc);
      out[o] = acc;
      if (zero_dp) a.dP[(size_t)c * nt + o] = 0.f;
    }
    __syncthreads();
  }
}

// Distinct rows: row[(jA, j3)] = sum_e P[c][jA, e] D_2[e] F_3[e, i3, j3, 0].
__global__ void ttm_rows_kernel(TtmArgs a) {
  extern __shared__ float sm[];
  const int r2 = a.r2, n3 = a.n3, nt = a.nA * r2;
  float* pt = sm;          // [nA][r2], times D_2
  float* f3 = pt + nt;     // [r2][n3]
  const int U = a.counts[0];
  for (int u = blockIdx.x; u < U; u += gridDim.x) {
    const int v = a.ulist[u];
    const int pr = v / a.m3, i3 = v - (v / a.m3) * a.m3;
    const int c = a.pos_pair[pr];
    const float* P = a.P + (size_t)c * nt;
    for (int o = threadIdx.x; o < nt; o += blockDim.x) pt[o] = P[o] * a.D2[o % r2];
    for (int o = threadIdx.x; o < r2 * n3; o += blockDim.x) {
      const int e = o / n3;
      f3[o] = a.F3[(e * a.m3 + i3) * n3 + (o - e * n3)];
    }
    __syncthreads();
    float* row = a.rows + (size_t)u * a.Dm;
    for (int j = threadIdx.x; j < a.Dm; j += blockDim.x) {
      const int jA = j / n3, j3 = j - (j / n3) * n3;
      float acc = 0.f;
      for (int e = 0; e < r2; ++e) acc = fmaf(pt[jA * r2 + e], f3[e * n3 + j3], acc);
      row[j] = acc;
    }
    __syncthreads();
  }
}

// out[b, :] = rows[upos[idx[b]], :], four floats at a time when Dm % 4 == 0.
__global__ void ttm_scatter_kernel(TtmArgs a, const int32_t* __restrict__ idx,
                                   float* __restrict__ out) {
  if ((a.Dm & 3) == 0) {
    const int q = a.Dm >> 2;
    const int64_t n = (int64_t)a.B * q;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
      const int b = (int)(i / q), j = (int)(i - (int64_t)b * q);
      const int v = idx[b];
      if (v < 0 || v >= a.V) continue;
      reinterpret_cast<float4*>(out)[i] =
          reinterpret_cast<const float4*>(a.rows)[(size_t)a.upos[v] * q + j];
    }
  } else {
    const int64_t n = (int64_t)a.B * a.Dm;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
      const int b = (int)(i / a.Dm), j = (int)(i - (int64_t)b * a.Dm);
      const int v = idx[b];
      if (v < 0 || v >= a.V) continue;
      out[i] = a.rows[(size_t)a.upos[v] * a.Dm + j];
    }
  }
}

// Backward unit w: the sum of up to kChunk occurrence rows of dout for one
// distinct row, into rows[w].
__global__ void ttm_chunk_sum_kernel(TtmArgs a, const float* __restrict__ dout) {
  const int C = a.counts[2];
  for (int w = blockIdx.x; w < C; w += gridDim.x) {
    const int u = a.unit_u[w];
    const int k = w - a.uoff[u];
    const int v = a.ulist[u];
    const int o0 = a.off[v] + k * kChunk;
    const int o1 = min(o0 + kChunk, a.off[v] + a.cnt[v]);
    float* dst = a.rows + (size_t)w * a.Dm;
    for (int j = threadIdx.x; j < a.Dm; j += blockDim.x) {
      float s = 0.f;
      for (int o = o0; o < o1; ++o) s += dout[(size_t)a.occ[o] * a.Dm + j];
      dst[j] = s;
    }
  }
}

// Per distinct row: dR = sum of its chunk sums; then
//   dF_3[e, i3, j3] += sum_jA P[c][jA, e] D_2[e] dR[jA, j3]
//   dP[c][jA, e]    += sum_j3 dR[jA, j3] F_3[e, i3, j3]
__global__ void ttm_row_grad_kernel(TtmArgs a, float* __restrict__ dF3) {
  extern __shared__ float sm[];
  const int r2 = a.r2, n3 = a.n3, nt = a.nA * r2, Dm = a.Dm;
  float* dR = sm;          // [Dm]
  float* pt = dR + Dm;     // [nA][r2], times D_2
  float* f3 = pt + nt;     // [r2][n3]
  const int U = a.counts[0];
  for (int u = blockIdx.x; u < U; u += gridDim.x) {
    const int v = a.ulist[u];
    const int pr = v / a.m3, i3 = v - (v / a.m3) * a.m3;
    const int c = a.pos_pair[pr];
    const int w0 = a.uoff[u], nch = (a.cnt[v] + kChunk - 1) / kChunk;
    for (int j = threadIdx.x; j < Dm; j += blockDim.x) {
      float s = 0.f;
      for (int w = w0; w < w0 + nch; ++w) s += a.rows[(size_t)w * Dm + j];
      dR[j] = s;
    }
    const float* P = a.P + (size_t)c * nt;
    for (int o = threadIdx.x; o < nt; o += blockDim.x) pt[o] = P[o] * a.D2[o % r2];
    for (int o = threadIdx.x; o < r2 * n3; o += blockDim.x) {
      const int e = o / n3;
      f3[o] = a.F3[(e * a.m3 + i3) * n3 + (o - e * n3)];
    }
    __syncthreads();
    for (int o = threadIdx.x; o < r2 * n3; o += blockDim.x) {
      const int e = o / n3, j3 = o - (o / n3) * n3;
      float acc = 0.f;
      for (int jA = 0; jA < a.nA; ++jA) acc = fmaf(pt[jA * r2 + e], dR[jA * n3 + j3], acc);
      atomicAdd(dF3 + (e * a.m3 + i3) * n3 + j3, acc);
    }
    float* dP = a.dP + (size_t)c * nt;
    for (int o = threadIdx.x; o < nt; o += blockDim.x) {
      const int jA = o / r2, e = o - (o / r2) * r2;
      float acc = 0.f;
      for (int j3 = 0; j3 < n3; ++j3) acc = fmaf(dR[jA * n3 + j3], f3[e * n3 + j3], acc);
      atomicAdd(dP + o, acc);
    }
    __syncthreads();
  }
}

// Per used prefix: back through P = F_1 D_1 F_2 and the D_2 scaling.
__global__ void ttm_pair_grad_kernel(TtmArgs a, float* __restrict__ dF1, float* __restrict__ dF2,
                                     float* __restrict__ dD1, float* __restrict__ dD2) {
  extern __shared__ float sm[];
  const int n1 = a.n1, n2 = a.n2, r1 = a.r1, r2 = a.r2, nt = a.nA * r2, w2 = n2 * r2;
  float* f1 = sm;             // [n1][r1] (without D_1)
  float* f2 = f1 + n1 * r1;   // [r1][n2][r2]
  float* G = f2 + r1 * w2;    // [nA][r2] gradient w.r.t. P
  float* H = G + nt;          // [n1][r1]
  const int Pn = a.counts[1];
  for (int c = blockIdx.x; c < Pn; c += gridDim.x) {
    const int p = a.plist[c];
    const int i1 = p / a.m2, i2 = p - (p / a.m2) * a.m2;
    for (int e = threadIdx.x; e < n1 * r1; e += blockDim.x) f1[e] = a.F1[i1 * n1 * r1 + e];
    for (int e = threadIdx.x; e < r1 * w2; e += blockDim.x) {
      const int b = e / w2;
      f2[e] = a.F2[(b * a.m2 + i2) * w2 + (e - b * w2)];
    }
    const float* dP = a.dP + (size_t)c * nt;
    for (int o = threadIdx.x; o < nt; o += blockDim.x) G[o] = dP[o] * a.D2[o % r2];
    __syncthreads();
    // dD_2[e] += sum_jA P[jA, e] dP[jA, e]
    const float* P = a.P + (size_t)c * nt;
    for (int e = threadIdx.x; e < r2; e += blockDim.x) {
      if (a.D2[e] == 0.f) continue;
      float acc = 0.f;
      for (int jA = 0; jA < a.nA; ++jA) acc = fmaf(P[jA * r2 + e], dP[jA * r2 + e], acc);
      atomicAdd(dD2 + e, acc);
    }
    // dF_2[b, i2, j2, e] += sum_j1 F_1[i1, j1, b] D_1[b] G[(j1, j2), e]
    for (int o = threadIdx.x; o < r1 * w2; o += blockDim.x) {
      const int b = o / w2, je = o - (o / w2) * w2;
      const float db = a.D1[b];
      float acc = 0.f;
      for (int j1 = 0; j1 < n1; ++j1) acc = fmaf(f1[j1 * r1 + b], G[j1 * w2 + je], acc);
      atomicAdd(dF2 + (b * a.m2 + i2) * w2 + je, acc * db);
    }
    // H[j1, b] = sum_{j2, e} G[(j1, j2), e] F_2[b, i2, j2, e]
    for (int o = threadIdx.x; o < n1 * r1; o += blockDim.x) {
      const int j1 = o / r1, b = o - (o / r1) * r1;
      float acc = 0.f;
      for (int je = 0; je < w2; ++je) acc = fmaf(G[j1 * w2 + je], f2[b * w2 + je], acc);
      H[o] = acc;
    }
    __syncthreads();
    // dF_1[0, i1, j1, b] += D_1[b] H[j1, b];  dD_1[b] += sum_j1 F_1[i1, j1, b] H[j1, b]
    for (int o = threadIdx.x; o < n1 * r1; o += blockDim.x)
      atomicAdd(dF1 + i1 * n1 * r1 + o, a.D1[o % r1] * H[o]);
    for (int b = threadIdx.x; b < r1; b += blockDim.x) {
      if (a.D1[b] == 0.f) continue;
      float acc = 0.f;
      for (int j1 = 0; j1 < n1; ++j1) acc = fmaf(f1[j1 * r1 + b], H[j1 * r1 + b], acc);
      atomicAdd(dD1 + b, acc);
    }
    __syncthreads();
  }
}

// ---- host side ---------------------------------------------------------------

struct TtmWs {
  size_t cnt, cursor, cnt_pair, off, upos, ulist, uoff, unit_u, pos_pair, plist, counts, occ, P,
      dP, rows, end;
  int64_t ucap, pcap, unit_cap;
  size_t zero_bytes;  // cnt .. cnt_pair, zeroed per call
};

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

TtmWs ttm_layout(const TtmPlan& P, int64_t B) {
  TtmWs w;
  w.ucap = std::min<int64_t>(B, P.V);
  w.pcap = std::min<int64_t>(B, P.npair);
  w.unit_cap = w.ucap + B / kChunk + 1;
  const int64_t nt = (int64_t)P.n[0] * P.n[1] * P.r[2];
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o = al(o + bytes);
    return r;
  };
  w.counts = take(16);  // first: the same offset for every batch size
  // cnt, cursor and cnt_pair are one zeroed block
  w.cnt = take(0);
  o = w.cnt + 4 * (size_t)P.V;
  w.cursor = o;
  o += 4 * (size_t)P.V;
  w.cnt_pair = o;
  o += 4 * (size_t)P.npair;
  w.zero_bytes = o - w.cnt;
  o = al(o);
  w.off = take(4 * (size_t)P.V);
  w.upos = take(4 * (size_t)P.V);
  w.ulist = take(4 * (size_t)w.ucap);
  w.uoff = take(4 * (size_t)w.ucap);
  w.unit_u = take(4 * (size_t)w.unit_cap);
  w.pos_pair = take(4 * (size_t)P.npair);
  w.plist = take(4 * (size_t)w.pcap);
  w.occ = take(4 * (size_t)B);
  w.P = take(4 * (size_t)(w.pcap * nt));
  w.dP = take(4 * (size_t)(w.pcap * nt));
  w.rows = take(4 * (size_t)(std::max(w.ucap, w.unit_cap) * P.Dm));
  w.end = o;
  return w;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

struct Units {
  float* one = nullptr;
  float* sink = nullptr;
};

bool unit_ptrs(Units* u) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_ttm_one) != cudaSuccess) return false;
  u->one = static_cast<float*>(p);
  if (cudaGetSymbolAddress(&p, g_ttm_sink) != cudaSuccess) return false;
  u->sink = static_cast<float*>(p);
  return true;
}

TtmArgs make_args(const TtmPlan& P, int64_t B, const float* params, void* ws, const TtmWs& w,
                  const Units& un) {
  TtmArgs a;
  a.B = (int)B;
  a.V = (int)P.V;
  a.npair = (int)P.npair;
  a.m1 = P.m[0]; a.m2 = P.m[1]; a.m3 = P.m[2];
  a.n1 = P.n[0]; a.n2 = P.n[1]; a.n3 = P.n[2];
  a.r1 = P.r[1]; a.r2 = P.r[2];
  a.nA = P.n[0] * P.n[1];
  a.Dm = (int)P.Dm;
  a.F1 = params + P.core_off[0];
  a.F2 = params + P.core_off[1];
  a.F3 = P.d == 3 ? params + P.core_off[2] : un.one;
  a.D1 = params + P.diag_off[0];
  a.D2 = P.d == 3 ? params + P.diag_off[1] : un.one;
  a.cnt = at<int>(ws, w.cnt);
  a.cursor = at<int>(ws, w.cursor);
  a.cnt_pair = at<int>(ws, w.cnt_pair);
  a.off = at<int>(ws, w.off);
  a.upos = at<int>(ws, w.upos);
  a.ulist = at<int>(ws, w.ulist);
  a.uoff = at<int>(ws, w.uoff);
  a.unit_u = at<int>(ws, w.unit_u);
  a.pos_pair = at<int>(ws, w.pos_pair);
  a.plist = at<int>(ws, w.plist);
  a.counts = at<int>(ws, w.counts);
  a.occ = at<int>(ws, w.occ);
  a.P = at<float>(ws, w.P);
  a.dP = at<float>(ws, w.dP);
  a.rows = at<float>(ws, w.rows);
  return a;
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

size_t pairs_smem(const TtmPlan& P) {
  return 4 * (size_t)(P.n[0] * P.r[1] + P.r[1] * P.n[1] * P.r[2]);
}
size_t rows_smem(const TtmPlan& P) {
  return 4 * (size_t)(P.n[0] * P.n[1] * P.r[2] + P.r[2] * P.n[2]);
}
size_t row_grad_smem(const TtmPlan& P) { return rows_smem(P) + 4 * (size_t)P.Dm; }
size_t pair_grad_smem(const TtmPlan& P) {
  return pairs_smem(P) + 4 * (size_t)(P.n[0] * P.n[1] * P.r[2] + P.n[0] * P.r[1]);
}

cudaError_t set_attrs() {
  static cudaError_t e = [] {
    const int big = kMaxSmemFloats * 4;
    cudaError_t r = cudaFuncSetAttribute(ttm_pairs_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(ttm_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(ttm_row_grad_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(ttm_pair_grad_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    return r;
  }();
  return e;
}

#define TTM_CUDA(call)                                 \
  do {                                                 \
    if ((call) != cudaSuccess) return TT_ERR_CUDA;     \
  } while (0)

// count, scan (and, for the backward, fill), pair products
tt_status ttm_prepare(const TtmPlan& P, int64_t B, const int32_t* idx, const TtmArgs& a,
                      const TtmWs& w, void* ws, bool backward, cudaStream_t st) {
  const int g = 2 * sm_count();
  TTM_CUDA(cudaMemsetAsync(at<char>(ws, w.cnt), 0, w.zero_bytes, st));
  int gb = (int)std::min<int64_t>((B + 255) / 256, 4 * sm_count());
  ttm_count_kernel<<<gb, 256, 0, st>>>(a, idx);
  ttm_scan_kernel<<<1, 1024, 0, st>>>(a);
  if (backward) ttm_fill_kernel<<<gb, 256, 0, st>>>(a, idx);
  ttm_pairs_kernel<<<g, 256, pairs_smem(P), st>>>(a, backward ? 1 : 0);
  count_launches(backward ? 4 : 3);
  TTM_CUDA(cudaGetLastError());
  return TT_OK;
}

}  // namespace

size_t ttm_workspace_bytes(const TtmPlan& P, int64_t B) { return ttm_layout(P, B).end; }

cudaError_t read_and_clear_ttm_status(DeviceStatus* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_ttm_status, sizeof(DeviceStatus));
  if (e != cudaSuccess) return e;
  DeviceStatus z{0, 0};
  return cudaMemcpyToSymbol(g_ttm_status, &z, sizeof(z));
}

}  // namespace ttc

using namespace ttc;

extern "C" {

tt_status tt_ttm_plan(const tt_ttm_desc* desc, tt_plan_t** out) {
  if (!out) return TT_ERR_INVALID_ARG;
  *out = nullptr;
  if (!desc || (desc->d != 2 && desc->d != 3)) return TT_ERR_INVALID_ARG;
  if (desc->flags & ~TT_ACCUMULATE) return TT_ERR_INVALID_ARG;
  const int d = desc->d;
  TtmPlan P;
  P.d = d;
  P.flags = desc->flags;
  int64_t V = 1, Dm = 1;
  for (int k = 0; k < d; ++k) {
    if (desc->row_modes[k] < 1 || desc->col_modes[k] < 1) return TT_ERR_INVALID_ARG;
    P.m[k] = desc->row_modes[k];
    P.n[k] = desc->col_modes[k];
    V *= P.m[k];
    Dm *= P.n[k];
    if (V > (1 << 24) || Dm > 8192) return TT_ERR_UNSUPPORTED;
  }
  if (desc->ranks[0] != 1 || desc->ranks[d] != 1) return TT_ERR_INVALID_ARG;
  for (int k = 1; k < d; ++k) {
    if (desc->ranks[k] < 1 || desc->ranks[k] > 4096) return TT_ERR_INVALID_ARG;
    if (desc->ranks[k] > 64) return TT_ERR_UNSUPPORTED;
    P.r[k] = desc->ranks[k];
  }
  P.V = V;
  P.Dm = Dm;
  P.npair = (int64_t)P.m[0] * P.m[1];
  size_t off = 0;
  for (int k = 0; k < d; ++k) {
    P.core_off[k] = off;
    off += (size_t)desc->ranks[k] * P.m[k] * P.n[k] * desc->ranks[k + 1];
  }
  for (int k = 1; k < d; ++k) {
    P.diag_off[k - 1] = off;
    off += (size_t)desc->ranks[k];
  }
  P.n_floats = off;
  // shared-memory tiles of the kernels
  if ((int64_t)P.n[0] * P.n[1] * P.r[2] > 8192 || (int64_t)P.r[1] * P.n[1] * P.r[2] > 16384 ||
      (int64_t)P.r[2] * P.n[2] > 8192 || pair_grad_smem(P) > 4 * (size_t)kMaxSmemFloats ||
      row_grad_smem(P) > 4 * (size_t)kMaxSmemFloats)
    return TT_ERR_UNSUPPORTED;
  tt_plan_s* p = new (std::nothrow) tt_plan_s();
  if (!p) return TT_ERR_INVALID_ARG;
  p->kind = 2;
  p->ttm = P;
  *out = p;
  return TT_OK;
}

tt_status tt_ttm_lookup(const tt_plan_t* plan, int64_t B, const int32_t* idx, const float* params,
                        float* out, void* ws, size_t ws_bytes, void* stream) {
  if (!plan || plan->kind != 2 || B < 0 || B > 0x7FFFFFFF) return TT_ERR_INVALID_ARG;
  if (B == 0) return TT_OK;
  if (!idx || !params || !out || (reinterpret_cast<uintptr_t>(out) & 15)) return TT_ERR_INVALID_ARG;
  const TtmPlan& P = plan->ttm;
  const TtmWs w = ttm_layout(P, B);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < w.end) return TT_ERR_WORKSPACE;
  Units un;
  if (set_attrs() != cudaSuccess || !unit_ptrs(&un)) return TT_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const TtmArgs a = make_args(P, B, params, ws, w, un);
  tt_status s = ttm_prepare(P, B, idx, a, w, ws, false, st);
  if (s != TT_OK) return s;
  const int g = 2 * sm_count();
  ttm_rows_kernel<<<g, 256, rows_smem(P), st>>>(a);
  ttm_scatter_kernel<<<4 * sm_count(), 256, 0, st>>>(a, idx, out);
  count_launches(2);
  return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

tt_status tt_ttm_lookup_backward(const tt_plan_t* plan, int64_t B, const int32_t* idx,
                                 const float* dout, const float* params, float* dparams,
                                 void* ws, size_t ws_bytes, void* stream) {
  if (!plan || plan->kind != 2 || B < 0 || B > 0x7FFFFFFF) return TT_ERR_INVALID_ARG;
  if (!params || !dparams) return TT_ERR_INVALID_ARG;
  const TtmPlan& P = plan->ttm;
  const bool acc = (P.flags & TT_ACCUMULATE) != 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!acc) TTM_CUDA(cudaMemsetAsync(dparams, 0, P.n_floats * sizeof(float), st));
  if (B == 0) return TT_OK;
  if (!idx || !dout) return TT_ERR_INVALID_ARG;
  const TtmWs w = ttm_layout(P, B);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < w.end) return TT_ERR_WORKSPACE;
  Units un;
  if (set_attrs() != cudaSuccess || !unit_ptrs(&un)) return TT_ERR_CUDA;
  const TtmArgs a = make_args(P, B, params, ws, w, un);
  tt_status s = ttm_prepare(P, B, idx, a, w, ws, true, st);
  if (s != TT_OK) return s;
  const int g = 2 * sm_count();
  float* dF1 = dparams + P.core_off[0];
  float* dF2 = dparams + P.core_off[1];
  float* dF3 = P.d == 3 ? dparams + P.core_off[2] : un.sink;
  float* dD1 = dparams + P.diag_off[0];
  float* dD2 = P.d == 3 ? dparams + P.diag_off[1] : un.sink + 32;
  ttm_chunk_sum_kernel<<<4 * sm_count(), 256, 0, st>>>(a, dout);
  ttm_row_grad_kernel<<<g, 256, row_grad_smem(P), st>>>(a, dF3);
  ttm_pair_grad_kernel<<<g, 256, pair_grad_smem(P), st>>>(a, dF1, dF2, dD1, dD2);
  count_launches(3);
  return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

tt_status tt_ttm_stats(const tt_plan_t* plan, const void* ws, int64_t* unique_rows,
                       int64_t* unique_pairs, void* stream) {
  if (!plan || plan->kind != 2 || !ws || !unique_rows || !unique_pairs) return TT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return TT_ERR_CUDA;
  int h[4] = {0, 0, 0, 0};  // the counts block opens the workspace
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return TT_ERR_CUDA;
  *unique_rows = h[0];
  *unique_pairs = h[1];
  return TT_OK;
}

}  // extern "C"
