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
// Forward:  count -> tiled scan -> per prefix: pair product and its rows ->
//           scatter.
// Backward: count -> tiled scan (+ row chunks) -> fill (occurrence lists) ->
//           chunk sums of dout -> per prefix: pair product, its rows' dF_3 and
//           pair-product gradient, then dF_1, dF_2, dD_1, dD_2.
// The per-row contractions of a prefix run as small dense GEMMs over batches
// of its used rows, register-blocked, from shared memory.
// Sums over repeated indices and over rows sharing a prefix use atomics.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>
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

// The bookkeeping kernels (count, tile sums, scan, tile write, fill) are
// launched with programmatic dependent launch: each waits for the grid
// before it in the stream (whose writes it may read) first thing, then lets
// the next grid start its own launch.  The per-prefix kernels and the row
// kernels are ordinary launches (measured slower with it).
__device__ __forceinline__ void ttm_pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
  float* rows;    // [ucap][Dm] distinct rows (forward) / [units][Dm] chunk sums (backward)
};

__global__ void ttm_count_kernel(TtmArgs a, const int32_t* __restrict__ idx) {
  ttm_pdl_enter();
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

// Inclusive scans over the block (a multiple of 32 threads, at most 1024)
// of three per-thread values (warp shuffles, then one warp over the warp
// totals).  After the call w1[nw-1], w2[nw-1], w3[nw-1] hold the block
// totals, nw = blockDim.x / 32.
__device__ void block_scan3(int& x1, int& x2, int& x3, int* w1, int* w2, int* w3) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 1; o < 32; o <<= 1) {
    const int y1 = __shfl_up_sync(0xffffffffu, x1, o);
    const int y2 = __shfl_up_sync(0xffffffffu, x2, o);
    const int y3 = __shfl_up_sync(0xffffffffu, x3, o);
    if (lane >= o) {
      x1 += y1;
      x2 += y2;
      x3 += y3;
    }
  }
  if (lane == 31) {
    w1[warp] = x1;
    w2[warp] = x2;
    w3[warp] = x3;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int v1 = lane < nw ? w1[lane] : 0, v2 = lane < nw ? w2[lane] : 0;
    int v3 = lane < nw ? w3[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int y1 = __shfl_up_sync(0xffffffffu, v1, o);
      const int y2 = __shfl_up_sync(0xffffffffu, v2, o);
      const int y3 = __shfl_up_sync(0xffffffffu, v3, o);
      if (lane >= o) {
        v1 += y1;
        v2 += y2;
        v3 += y3;
      }
    }
    if (lane < nw) {
      w1[lane] = v1;
      w2[lane] = v2;
      w3[lane] = v3;
    }
  }
  __syncthreads();
  if (warp > 0) {
    x1 += w1[warp - 1];
    x2 += w2[warp - 1];
    x3 += w3[warp - 1];
  }
}

constexpr int kScanPer = 8;                    // elements per thread of a tile
constexpr int kScanThreads = 256;
constexpr int kScanTile = kScanThreads * kScanPer;

// Per-thread sums over its kScanPer consecutive entries of a tile: rows give
// (occurrences, distinct, backward units), prefixes give (used, 0, 0).
__device__ void tile_sums(const TtmArgs& a, bool rows, int base, int n, int* c, int* f, int* u) {
  const int lo = threadIdx.x * kScanPer, hi = min(lo + kScanPer, n);
  *c = *f = *u = 0;
  for (int i = lo; i < hi; ++i) {
    const int x = rows ? a.cnt[base + i] : a.cnt_pair[base + i];
    if (rows) {
      *c += x;
      *f += x > 0;
      *u += (x + kChunk - 1) / kChunk;
    } else {
      *c += x != 0;
    }
  }
}

// Blocks [0, ntr) cover row tiles, [ntr, ntr + ntp) prefix tiles: each
// writes its tile totals (tsum[3 * tile + 0..2]).
__global__ void __launch_bounds__(kScanThreads) ttm_tile_sum_kernel(TtmArgs a, int ntr, int* tsum) {
  ttm_pdl_enter();
  __shared__ int w1[32], w2[32], w3[32];
  const bool rows = (int)blockIdx.x < ntr;
  const int tile = rows ? blockIdx.x : blockIdx.x - ntr;
  const int base = tile * kScanTile;
  const int n = min(kScanTile, (rows ? a.V : a.npair) - base);
  int c, f, u;
  tile_sums(a, rows, base, n, &c, &f, &u);
  block_scan3(c, f, u, w1, w2, w3);
  if (threadIdx.x == 0) {
    const int nw = blockDim.x >> 5;
    tsum[3 * blockIdx.x + 0] = w1[nw - 1];
    tsum[3 * blockIdx.x + 1] = w2[nw - 1];
    tsum[3 * blockIdx.x + 2] = w3[nw - 1];
  }
}

// One block: exclusive prefix of the tile totals (rows and prefixes apart);
// the grand totals go to counts[0..2].
__global__ void __launch_bounds__(1024) ttm_tile_scan_kernel(TtmArgs a, int ntr, int ntp, int* tsum) {
  ttm_pdl_enter();
  __shared__ int w1[32], w2[32], w3[32];
  for (int part = 0; part < 2; ++part) {
    const int t0 = part == 0 ? 0 : ntr, nt = part == 0 ? ntr : ntp;
    int carry_c = 0, carry_f = 0, carry_u = 0;
    for (int base = 0; base < nt; base += 1024) {
      const int i = base + threadIdx.x;
      int c = 0, f = 0, u = 0;
      if (i < nt) {
        c = tsum[3 * (t0 + i)];
        f = tsum[3 * (t0 + i) + 1];
        u = tsum[3 * (t0 + i) + 2];
      }
      int ic = c, iff = f, iu = u;
      block_scan3(ic, iff, iu, w1, w2, w3);
      if (i < nt) {
        tsum[3 * (t0 + i)] = carry_c + ic - c;
        tsum[3 * (t0 + i) + 1] = carry_f + iff - f;
        tsum[3 * (t0 + i) + 2] = carry_u + iu - u;
      }
      carry_c += w1[31];
      carry_f += w2[31];
      carry_u += w3[31];
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      if (part == 0) {
        a.counts[0] = carry_f;
        a.counts[2] = carry_u;
      } else {
        a.counts[1] = carry_c;
      }
    }
  }
}

// Rescans each tile from its offset and writes: rows -> occurrence offsets,
// distinct slots, row list, first backward unit and the unit list; prefixes
// -> prefix slots and the prefix list.
__global__ void __launch_bounds__(kScanThreads) ttm_tile_write_kernel(TtmArgs a, int ntr,
                                                                     const int* tsum) {
  ttm_pdl_enter();
  __shared__ int w1[32], w2[32], w3[32];
  const bool rows = (int)blockIdx.x < ntr;
  const int tile = rows ? blockIdx.x : blockIdx.x - ntr;
  const int base = tile * kScanTile;
  const int n = min(kScanTile, (rows ? a.V : a.npair) - base);
  int c, f, u;
  tile_sums(a, rows, base, n, &c, &f, &u);
  int ic = c, iff = f, iu = u;
  block_scan3(ic, iff, iu, w1, w2, w3);
  const int* off = tsum + 3 * blockIdx.x;
  int ec = off[0] + ic - c, ef = off[1] + iff - f, eu = off[2] + iu - u;
  const int lo = threadIdx.x * kScanPer, hi = min(lo + kScanPer, n);
  for (int i = lo; i < hi; ++i) {
    const int v = base + i;
    if (rows) {
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
    } else if (a.cnt_pair[v]) {
      a.pos_pair[v] = ec;
      a.plist[ec++] = v;
    }
  }
}

// Occurrence lists: occ[off[v] ..] = the positions b with idx[b] == v.  A
// position beyond the row's count (counts of another batch, kept in the
// workspace by a lookup whose indices differ: a broken TT_REUSE_MERGE
// promise) is not written, and the status word records the error.
__global__ void ttm_fill_kernel(TtmArgs a, const int32_t* __restrict__ idx) {
  ttm_pdl_enter();
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < a.B; b += gridDim.x * blockDim.x) {
    const int v = idx[b];
    if (v < 0 || v >= a.V) continue;
    const int k = atomicAdd(a.cursor + v, 1);
    if (k < a.cnt[v])
      a.occ[a.off[v] + k] = b;
    else
      ttm_error(3);
  }
}

// Asynchronous 4-byte global -> shared copies: a thread issues all of its
// staging copies before waiting, so a staging pass costs one round trip
// instead of one per element.
__device__ __forceinline__ void cp_async4(float* smem, const float* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<unsigned>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

constexpr int kRowBatch = 5;  // used rows of a prefix handled together (4 blocks an SM fit)

// Shared-memory row pitches chosen against bank conflicts: an odd pitch for
// the F_2 slice rows (read across rows by the H product, scalar loads); for
// tiles read four floats at a time along their rows, a multiple of 4 whose
// quarter is odd, so that the 16-byte reads of eight consecutive rows fall on
// eight different bank quads; and a dR row pitch congruent to n3 mod 32, so
// that consecutive (row, j3) columns fall in consecutive banks.
__host__ __device__ inline int f2_pitch(int n2, int r2) { return (n2 * r2) | 1; }
__host__ __device__ inline int pad4(int x) { return (x + 3) & ~3; }
__host__ __device__ inline int vec_pitch(int x) {
  const int p = pad4(x);
  return (p / 4) % 2 ? p : p + 4;
}
__host__ __device__ inline int dr_pitch(int Dm, int n3) {
  return Dm + (((n3 - Dm) % 32) + 32) % 32;
}

// Shared-memory tiles (float offsets, each start a multiple of 4) of the
// per-prefix kernels:
//   f1 [n1][r1] | f2 [r1][n2 r2] pitch F2P | pt [n1 n2][PTP] (P; columns
//   r2 .. K2P-1 zero) | forward: f3 [kRowBatch n3][F3P] (F_3 slices, e along
//   the rows; columns r2 .. K2P-1 zero) | backward: dP [n1 n2][r2], H [n1][r1],
//   dR [kRowBatch][DP], f3 [r2][F3P] (e down the rows)
struct TtmSmem {
  int F2P, PTP, K2P, F3P, DP;
  int f1, f2, pt, dP, H, dR, f3, total;
};
__host__ __device__ inline TtmSmem ttm_smem(int n1, int n2, int n3, int r1, int r2, int Dm,
                                            bool backward) {
  TtmSmem t;
  t.F2P = f2_pitch(n2, r2);
  t.K2P = pad4(r2);
  t.PTP = vec_pitch(r2);
  t.F3P = backward ? vec_pitch(kRowBatch * n3) : vec_pitch(r2);
  t.DP = dr_pitch(Dm, n3);
  int o = 0;
  t.f1 = o; o = pad4(o + n1 * r1);
  t.f2 = o; o = pad4(o + r1 * t.F2P);
  t.pt = o; o = pad4(o + n1 * n2 * t.PTP);
  t.dP = t.H = t.dR = 0;
  if (backward) {
    t.dP = o; o = pad4(o + n1 * n2 * r2);
    t.H = o; o = pad4(o + n1 * r1);
    t.dR = o; o = pad4(o + kRowBatch * t.DP);
    t.f3 = o; o = pad4(o + r2 * t.F3P);
  } else {
    t.f3 = o; o = pad4(o + kRowBatch * n3 * t.F3P);
  }
  t.total = o;
  return t;
}

// Stages F_1[0, i1] (times D_1 when scale_d1) and F_2[:, i2] for prefix p,
// and computes the pair product P[(j1, j2), e] = sum_b F_1[0, i1, j1, b] D_1[b]
// F_2[b, i2, j2, e] into pt (times D_2[e] when scale_d2).  Ends synchronised.
__device__ void ttm_pair_product(const TtmArgs& a, int p, float* f1, float* f2, float* pt,
                                 int PTP, bool scale_d1, bool scale_d2) {
  const int n1 = a.n1, n2 = a.n2, r1 = a.r1, r2 = a.r2, w2 = n2 * r2;
  const int F2P = f2_pitch(n2, r2);
  const int i1 = p / a.m2, i2 = p - (p / a.m2) * a.m2;
  for (int e = threadIdx.x; e < n1 * r1; e += blockDim.x) cp_async4(f1 + e, a.F1 + i1 * n1 * r1 + e);
  for (int b = 0; b < r1; ++b) {  // row b of the slice is contiguous in F_2
    const float* src = a.F2 + (b * a.m2 + i2) * w2;
    for (int e = threadIdx.x; e < w2; e += blockDim.x) cp_async4(f2 + b * F2P + e, src + e);
  }
  cp_async_wait_all();
  __syncthreads();
  // one thread per column (j2, e) of F_2's slice; up to 8 rows j1 at a time
  // in registers, so each loaded F_2 value serves 8 products
  for (int je = threadIdx.x; je < w2; je += blockDim.x) {
    const int j2 = je / r2, e = je - j2 * r2;
    float* dst = pt + j2 * PTP + e;          // P[(j1, j2), e] at ((j1 n2 + j2) PTP + e)
    const float d2 = scale_d2 ? a.D2[e] : 1.f;
    for (int j0 = 0; j0 < n1; j0 += 8) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int b = 0; b < r1; ++b) {
        const float y = f2[b * F2P + je] * (scale_d1 ? a.D1[b] : 1.f);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (j0 + i < n1) acc[i] = fmaf(f1[(j0 + i) * r1 + b], y, acc[i]);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (j0 + i < n1) dst[(j0 + i) * n2 * PTP] = acc[i] * d2;
    }
  }
  __syncthreads();
}

// The used rows of prefix p (i3 with cnt[p m3 + i3] > 0) in increasing i3,
// into list[0, *n), for i3 in [base, base + 256); ends synchronised.
__device__ void used_rows(const TtmArgs& a, int p, int base, int* list, int* n) {
  __shared__ int wc[8];
  const int i3 = base + (int)threadIdx.x;
  const bool use = threadIdx.x < 256 && i3 < a.m3 && a.cnt[p * a.m3 + i3] > 0;
  const unsigned m = __ballot_sync(0xffffffffu, use);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0 && warp < 8) wc[warp] = __popc(m);
  __syncthreads();
  int before = 0, total = 0;
  for (int w = 0; w < 8; ++w) {
    if (w < warp) before += wc[w];
    total += wc[w];
  }
  if (use) list[before + __popc(m & ((1u << lane) - 1u))] = i3;
  if (threadIdx.x == 0) *n = total;
  __syncthreads();
}

// C(m, n) = sum_k A(m, k) B(k, n) for one block, operands in shared memory,
// each thread holding a 4 x 4 tile of C in registers (8 loads feed 16 FMAs).
// K runs as k1 < K1 outer, k2 < K2 inner:
//   A(m, k1, k2) = A[m am + k1 ak1 + k2 ak2]
//   B(k1, k2, n) = B[(n / nq) bq + (n % nq) bn + k1 bk1 + k2 bk2]
// A thread's rows are m_t, m_t + TM, ... and its columns n_t, n_t + TN, ...
// (TM, TN: thread rows and columns), so the lanes of a warp read consecutive
// columns.  epi(m, n, c) receives every output once.
struct BlockGemm {
  int M, N, K1, K2;
  int am, ak1, ak2;
  int nq, bq, bn, bk1, bk2;
};

template <typename Epi>
__device__ void block_gemm(const float* __restrict__ A, const float* __restrict__ B,
                           const BlockGemm& g, Epi epi) {
  const int TM = (g.M + 3) >> 2, TN = (g.N + 3) >> 2;
  for (int t = threadIdx.x; t < TM * TN; t += blockDim.x) {
    const int mt = t / TN, nt = t - mt * TN;
    int ao[4], bo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = mt + i * TM;
      ao[i] = (m < g.M ? m : 0) * g.am;
      const int n0 = nt + i * TN, n = n0 < g.N ? n0 : 0;
      const int q = n / g.nq;
      bo[i] = q * g.bq + (n - q * g.nq) * g.bn;
    }
    float acc[4][4] = {};
    for (int k1 = 0; k1 < g.K1; ++k1) {
      const float* a1 = A + k1 * g.ak1;
      const float* b1 = B + k1 * g.bk1;
      for (int k2 = 0; k2 < g.K2; ++k2) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          av[i] = a1[ao[i] + k2 * g.ak2];
          bv[i] = b1[bo[i] + k2 * g.bk2];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[i][c] = fmaf(av[i], bv[c], acc[i][c]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (mt + i * TM < g.M && nt + c * TN < g.N) epi(mt + i * TM, nt + c * TN, acc[i][c]);
  }
}


// block_gemm for operands read four floats at a time along K: K2 a multiple
// of 4, ak2 = bk2 = 1, every other stride a multiple of 4 and A, B 16-byte
// aligned.
template <typename Epi>
__device__ void block_gemm4(const float* __restrict__ A, const float* __restrict__ B,
                            const BlockGemm& g, Epi epi) {
  const int TM = (g.M + 3) >> 2, TN = (g.N + 3) >> 2;
  for (int t = threadIdx.x; t < TM * TN; t += blockDim.x) {
    const int mt = t / TN, nt = t - mt * TN;
    int ao[4], bo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = mt + i * TM;
      ao[i] = (m < g.M ? m : 0) * g.am;
      const int n0 = nt + i * TN, n = n0 < g.N ? n0 : 0;
      const int q = n / g.nq;
      bo[i] = q * g.bq + (n - q * g.nq) * g.bn;
    }
    float acc[4][4] = {};
    for (int k1 = 0; k1 < g.K1; ++k1) {
      const float* a1 = A + k1 * g.ak1;
      const float* b1 = B + k1 * g.bk1;
      for (int k2 = 0; k2 < g.K2; k2 += 4) {
        float4 av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          av[i] = *reinterpret_cast<const float4*>(a1 + ao[i] + k2);
          bv[i] = *reinterpret_cast<const float4*>(b1 + bo[i] + k2);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float x = acc[i][c];
            x = fmaf(av[i].x, bv[c].x, x);
            x = fmaf(av[i].y, bv[c].y, x);
            x = fmaf(av[i].z, bv[c].z, x);
            x = fmaf(av[i].w, bv[c].w, x);
            acc[i][c] = x;
          }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (mt + i * TM < g.M && nt + c * TN < g.N) epi(mt + i * TM, nt + c * TN, acc[i][c]);
  }
}

// f3t[k n3 + j3][e] = F_3[e, i3_k, j3] for the kb rows i3_k of a batch (e
// along the rows, pitch F3P); ends with the copies landed.
__device__ void stage_f3t(const TtmArgs& a, const int* i3s, int kb, float* f3t, int F3P) {
  const int n3 = a.n3, w = kb * n3;
  for (int o = threadIdx.x; o < a.r2 * w; o += blockDim.x) {
    const int e = o / w, rem = o - e * w;
    const int k = rem / n3, j3 = rem - k * n3;
    cp_async4(f3t + rem * F3P + e, a.F3 + (e * a.m3 + i3s[k]) * n3 + j3);
  }
  cp_async_wait_all();
}

// f3b[e][k n3 + j3] = F_3[e, i3_k, j3] for the kb rows i3_k of a batch (each
// (e, k) run of n3 floats is contiguous in F_3); ends with the copies landed
// (the caller synchronises the block).
__device__ void stage_f3(const TtmArgs& a, const int* i3s, int kb, float* f3b, int FP) {
  const int n3 = a.n3, runs = a.r2 * kb;
  for (int o = threadIdx.x; o < runs * n3; o += blockDim.x) {
    const int run = o / n3, j3 = o - run * n3;
    const int e = run / kb, k = run - e * kb;
    cp_async4(f3b + e * FP + k * n3 + j3, a.F3 + (e * a.m3 + i3s[k]) * n3 + j3);
  }
  cp_async_wait_all();
}

// Forward, one block of 256 threads per used prefix (slot c): its pair
// product P (with D_2) in shared memory, then its used rows kRowBatch at a
// time as one block GEMM read four floats at a time,
//   row_k[(jA, j3)] = sum_e P[jA, e] F_3[e, i3_k, j3]  ->  rows[upos[v_k]],
// with M = n1 n2, N = (rows of the batch) n3, K = r2 padded with zeros to a
// multiple of 4.
__global__ void __launch_bounds__(256, 4) ttm_pair_rows_kernel(TtmArgs a) {
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  __shared__ int list[256];
  __shared__ int nlist;
  __shared__ long long rbase[kRowBatch];
  const int n3 = a.n3, r2 = a.r2;
  const TtmSmem L = ttm_smem(a.n1, a.n2, n3, a.r1, r2, a.Dm, false);
  const int c = blockIdx.x;
  if (c >= a.counts[1]) return;
  float* f1 = sm + L.f1;
  float* f2 = sm + L.f2;
  float* pt = sm + L.pt;                    // [nA][PTP], D_1 inside, times D_2
  float* f3t = sm + L.f3;                   // [kRowBatch n3][F3P]: F_3[:, i3_k, j3] along rows
  // the K padding columns r2 .. K2P-1 of P and of the F_3 slices stay zero
  const int padw = L.K2P - r2;
  for (int o = threadIdx.x; o < a.nA * padw; o += blockDim.x)
    pt[(o / padw) * L.PTP + r2 + o % padw] = 0.f;
  for (int o = threadIdx.x; o < kRowBatch * n3 * padw; o += blockDim.x)
    f3t[(o / padw) * L.F3P + r2 + o % padw] = 0.f;
  const int p = a.plist[c];
  ttm_pair_product(a, p, f1, f2, pt, L.PTP, true, true);  // ends synchronised
  for (int base = 0; base < a.m3; base += 256) {
    used_rows(a, p, base, list, &nlist);
    for (int k0 = 0; k0 < nlist; k0 += kRowBatch) {
      const int kb = min(kRowBatch, nlist - k0);
      if ((int)threadIdx.x < kb)
        rbase[threadIdx.x] = (long long)a.upos[p * a.m3 + list[k0 + threadIdx.x]] * a.Dm;
      stage_f3t(a, list + k0, kb, f3t, L.F3P);
      __syncthreads();
      BlockGemm g;
      g.M = a.nA; g.N = kb * n3; g.K1 = 1; g.K2 = L.K2P;
      g.am = L.PTP; g.ak1 = 0; g.ak2 = 1;
      g.nq = 1 << 30; g.bq = 0; g.bn = L.F3P; g.bk1 = 0; g.bk2 = 1;
      float* rows = a.rows;
      block_gemm4(pt, f3t, g, [&](int jA, int n, float v) {
        const int k = n / n3;
        rows[rbase[k] + jA * n3 + (n - k * n3)] = v;
      });
      __syncthreads();  // f3t and rbase are refilled next
    }
  }
}

// out[b, :] = rows[upos[idx[b]], :]: one warp per index (one lookup of its
// row), the lanes copying the row four floats at a time when Dm % 4 == 0.
__global__ void ttm_scatter_kernel(TtmArgs a, const int32_t* __restrict__ idx,
                                   float* __restrict__ out) {
  const int lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
  for (int b = blockIdx.x * wpb + (threadIdx.x >> 5); b < a.B; b += gridDim.x * wpb) {
    const int v = idx[b];
    if (v < 0 || v >= a.V) continue;
    const size_t src = (size_t)a.upos[v] * a.Dm, dst = (size_t)b * a.Dm;
    if ((a.Dm & 3) == 0) {
      const float4* s4 = reinterpret_cast<const float4*>(a.rows + src);
      float4* d4 = reinterpret_cast<float4*>(out + dst);
      for (int j = lane; j < (a.Dm >> 2); j += 32) d4[j] = s4[j];
    } else {
      for (int j = lane; j < a.Dm; j += 32) out[dst + j] = a.rows[src + j];
    }
  }
}

// Backward unit w: the sum of up to kChunk occurrence rows of dout for one
// distinct row, into rows[w].  The occurrence list goes to shared memory
// first so that all of a thread's loads are independent.
__global__ void __launch_bounds__(256) ttm_chunk_sum_kernel(TtmArgs a,
                                                            const float* __restrict__ dout) {
  __shared__ int ob[kChunk];
  const int w = blockIdx.x;
  if (w >= a.counts[2]) return;
  const int u = a.unit_u[w];
  const int k = w - a.uoff[u];
  const int v = a.ulist[u];
  const int o0 = a.off[v] + k * kChunk;
  const int n = min(kChunk, a.off[v] + a.cnt[v] - o0);
  if ((int)threadIdx.x < n) {
    int b = a.occ[o0 + threadIdx.x];
    if ((unsigned)b >= (unsigned)a.B) {  // a list left unfilled (a broken reuse promise)
      ttm_error(4);
      b = 0;
    }
    ob[threadIdx.x] = b;
  }
  __syncthreads();
  if ((a.Dm & 3) == 0) {
    const int q = a.Dm >> 2;
    const float4* src = reinterpret_cast<const float4*>(dout);
    float4* dst = reinterpret_cast<float4*>(a.rows) + (size_t)w * q;
    for (int j = threadIdx.x; j < q; j += blockDim.x) {
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
      for (int o = 0; o < n; ++o) {
        const float4 x = src[(size_t)ob[o] * q + j];
        s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
      }
      dst[j] = s;
    }
  } else {
    float* dst = a.rows + (size_t)w * a.Dm;
    for (int j = threadIdx.x; j < a.Dm; j += blockDim.x) {
      float s = 0.f;
#pragma unroll 8
      for (int o = 0; o < n; ++o) s += dout[(size_t)ob[o] * a.Dm + j];
      dst[j] = s;
    }
  }
}

// Backward, one block of 256 threads per used prefix (slot c).  Its used
// rows, kRowBatch at a time: dR_k = the sum of row k's chunk sums, then two
// block GEMMs over the batch,
//   dF_3[e, i3_k, j3] += D_2[e] sum_jA P[jA, e] dR_k[jA, j3]   (P without D_2)
//   dP[jA, e]         += sum_{k, j3} dR_k[jA, j3] F_3[e, i3_k, j3]
// then back through P D_2 = F_1 D_1 F_2 D_2 for this prefix:
//   dD_2[e] += sum_jA P[jA, e] dP[jA, e];  G = dP D_2
//   dF_2[b, i2, j2, e] += D_1[b] sum_j1 F_1[i1, j1, b] G[(j1, j2), e]
//   H[j1, b] = sum_{j2, e} G[(j1, j2), e] F_2[b, i2, j2, e]
//   dF_1[0, i1, j1, b] += D_1[b] H[j1, b];  dD_1[b] += sum_j1 F_1[i1, j1, b] H[j1, b]
// (dD entries of pruned ranks, D == 0, stay untouched).
__global__ void __launch_bounds__(256, 4) ttm_pair_backward_kernel(TtmArgs a, float* __restrict__ dF1,
                                                                float* __restrict__ dF2,
                                                                float* __restrict__ dF3,
                                                                float* __restrict__ dD1,
                                                                float* __restrict__ dD2) {
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  __shared__ int list[256];
  __shared__ int nlist;
  __shared__ int ri3[kRowBatch], rw0[kRowBatch], rnch[kRowBatch];
  const int n1 = a.n1, n2 = a.n2, n3 = a.n3, r1 = a.r1, r2 = a.r2;
  const int w2 = n2 * r2, nt = a.nA * r2, Dm = a.Dm;
  const TtmSmem L = ttm_smem(n1, n2, n3, r1, r2, Dm, true);
  const int FP = L.F3P, F2P = L.F2P, DP = L.DP, PTP = L.PTP;
  const int c = blockIdx.x;
  if (c >= a.counts[1]) return;
  float* f1 = sm + L.f1;    // [n1][r1] (without D_1)
  float* f2 = sm + L.f2;    // [r1][n2 r2], row pitch F2P
  float* pt = sm + L.pt;    // [nA][PTP] (D_1 inside, without D_2)
  float* dP = sm + L.dP;    // [nA][r2]
  float* H = sm + L.H;      // [n1][r1]
  float* dRb = sm + L.dR;   // [kRowBatch][Dm], row pitch DP
  float* f3b = sm + L.f3;   // [r2][kRowBatch n3], row pitch FP
  // the dP product reads four floats at a time along (k, j3) when n3 allows
  const bool vec = n3 % 4 == 0;
  const int p = a.plist[c];
  const int i1 = p / a.m2, i2 = p - (p / a.m2) * a.m2;
  for (int o = threadIdx.x; o < nt; o += blockDim.x) dP[o] = 0.f;
  ttm_pair_product(a, p, f1, f2, pt, PTP, true, false);
  for (int base = 0; base < a.m3; base += 256) {
    used_rows(a, p, base, list, &nlist);
    for (int k0 = 0; k0 < nlist; k0 += kRowBatch) {
      const int kb = min(kRowBatch, nlist - k0);
      if ((int)threadIdx.x < kb) {
        const int i3 = list[k0 + threadIdx.x], v = p * a.m3 + i3;
        ri3[threadIdx.x] = i3;
        rw0[threadIdx.x] = a.uoff[a.upos[v]];
        rnch[threadIdx.x] = (a.cnt[v] + kChunk - 1) / kChunk;
      }
      __syncthreads();
      // dR_k: the first chunk sum copied asynchronously, further chunks
      // (rows seen more than kChunk times) added after it has landed
      for (int k = 0; k < kb; ++k) {
        const float* src = a.rows + (size_t)rw0[k] * Dm;
        for (int j = threadIdx.x; j < Dm; j += blockDim.x) cp_async4(dRb + k * DP + j, src + j);
      }
      stage_f3(a, ri3, kb, f3b, FP);
      __syncthreads();
      for (int k = 0; k < kb; ++k) {
        if (rnch[k] <= 1) continue;
        const float* src = a.rows + (size_t)rw0[k] * Dm;
        for (int j = threadIdx.x; j < Dm; j += blockDim.x) {
          float sacc = dRb[k * DP + j];
          for (int w = 1; w < rnch[k]; ++w) sacc += src[(size_t)w * Dm + j];
          dRb[k * DP + j] = sacc;
        }
      }
      __syncthreads();
      BlockGemm g3;  // dF_3 slices: M = r2 (e), N = kb n3 ((k, j3)), K = nA
      g3.M = r2; g3.N = kb * n3; g3.K1 = 1; g3.K2 = a.nA;
      g3.am = 1; g3.ak1 = 0; g3.ak2 = PTP;
      g3.nq = n3; g3.bq = DP; g3.bn = 1; g3.bk1 = 0; g3.bk2 = n3;
      const float* D2 = a.D2;
      const int m3 = a.m3;
      block_gemm(pt, dRb, g3, [&](int e, int n, float v) {
        const int k = n / n3;
        atomicAdd(dF3 + (e * m3 + ri3[k]) * n3 + (n - k * n3), v * D2[e]);
      });
      BlockGemm gp;  // dP: M = nA (jA), N = r2 (e), K = (k, j3)
      gp.M = a.nA; gp.N = r2; gp.K1 = kb; gp.K2 = n3;
      gp.am = n3; gp.ak1 = DP; gp.ak2 = 1;
      gp.nq = 1 << 30; gp.bq = 0; gp.bn = FP; gp.bk1 = n3; gp.bk2 = 1;
      // every dP entry has one owner thread (the same in every batch)
      auto add_dp = [&](int jA, int e, float v) { dP[jA * r2 + e] += v; };
      if (vec)
        block_gemm4(dRb, f3b, gp, add_dp);
      else
        block_gemm(dRb, f3b, gp, add_dp);
      __syncthreads();  // dRb, f3b and the row metadata are refilled next
    }
  }
  for (int e = threadIdx.x; e < r2; e += blockDim.x) {
    if (a.D2[e] == 0.f) continue;
    float acc = 0.f;
    for (int jA = 0; jA < a.nA; ++jA) acc = fmaf(pt[jA * PTP + e], dP[jA * r2 + e], acc);
    atomicAdd(dD2 + e, acc);
  }
  __syncthreads();
  for (int o = threadIdx.x; o < nt; o += blockDim.x) dP[o] *= a.D2[o % r2];  // G
  __syncthreads();
  // dF_2: one thread per column (j2, e), G's column in registers (8 rows j1
  // at a time)
  for (int je = threadIdx.x; je < w2; je += blockDim.x) {
    float* dst = dF2 + i2 * w2 + je;
    for (int j0 = 0; j0 < n1; j0 += 8) {
      float g[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = j0 + i < n1 ? dP[(j0 + i) * w2 + je] : 0.f;
      for (int b = 0; b < r1; ++b) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (j0 + i < n1) acc = fmaf(f1[(j0 + i) * r1 + b], g[i], acc);
        atomicAdd(dst + b * a.m2 * w2, acc * a.D1[b]);
      }
    }
  }
  for (int o = threadIdx.x; o < n1 * r1; o += blockDim.x) {
    const int j1 = o / r1, b = o - (o / r1) * r1;
    float acc = 0.f;
    for (int je = 0; je < w2; ++je) acc = fmaf(dP[j1 * w2 + je], f2[b * F2P + je], acc);
    H[o] = acc;
  }
  __syncthreads();
  for (int o = threadIdx.x; o < n1 * r1; o += blockDim.x)
    atomicAdd(dF1 + i1 * n1 * r1 + o, a.D1[o % r1] * H[o]);
  for (int b = threadIdx.x; b < r1; b += blockDim.x) {
    if (a.D1[b] == 0.f) continue;
    float acc = 0.f;
    for (int j1 = 0; j1 < n1; ++j1) acc = fmaf(f1[j1 * r1 + b], H[j1 * r1 + b], acc);
    atomicAdd(dD1 + b, acc);
  }
}

// ---- host side ---------------------------------------------------------------

struct TtmWs {
  size_t cnt, cursor, cnt_pair, off, upos, ulist, uoff, unit_u, pos_pair, plist, counts, occ,
      tsum, rows, end;
  int64_t ucap, pcap, unit_cap;
  int ntr, ntp;  // scan tiles over the rows and over the prefixes
  size_t zero_bytes;  // cnt .. cnt_pair, zeroed per call
};

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

TtmWs ttm_layout(const TtmPlan& P, int64_t B) {
  TtmWs w;
  w.ucap = std::min<int64_t>(B, P.V);
  w.pcap = std::min<int64_t>(B, P.npair);
  w.unit_cap = w.ucap + B / kChunk + 1;
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
  w.ntr = (int)((P.V + kScanTile - 1) / kScanTile);
  w.ntp = (int)((P.npair + kScanTile - 1) / kScanTile);
  w.tsum = take(4 * 3 * (size_t)(w.ntr + w.ntp));
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

// Device addresses of the unit core and the sink, looked up once per device
// (the first call on a device should come before any stream capture).
bool unit_ptrs(Units* u) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static Units cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev].one) {
    void* p = nullptr;
    void* q = nullptr;
    if (cudaGetSymbolAddress(&p, g_ttm_one) != cudaSuccess ||
        cudaGetSymbolAddress(&q, g_ttm_sink) != cudaSuccess)
      return false;
    cache[dev].one = static_cast<float*>(p);
    cache[dev].sink = static_cast<float*>(q);
  }
  *u = cache[dev];
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

// Dynamic shared memory (bytes) of the per-prefix kernels.
size_t pair_rows_smem(const TtmPlan& P) {
  return 4 * (size_t)ttm_smem(P.n[0], P.n[1], P.n[2], P.r[1], P.r[2], (int)P.Dm, false).total;
}
size_t pair_backward_smem(const TtmPlan& P) {
  return 4 * (size_t)ttm_smem(P.n[0], P.n[1], P.n[2], P.r[1], P.r[2], (int)P.Dm, true).total;
}

cudaError_t set_attrs() {
  static PerDevice once;
  return once.get([] {
    const int big = kMaxSmemFloats * 4;
    cudaError_t r = cudaFuncSetAttribute(ttm_pair_rows_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(ttm_pair_backward_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    // all of the unified L1 / shared memory as shared memory, so that several
    // blocks of these kernels fit an SM
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(ttm_pair_rows_kernel,
                               cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(ttm_pair_backward_kernel,
                               cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    return r;
  });
}

bool ttm_pdl_on() {
  static int on = -1;
  if (on < 0) {
    const char* e = getenv("TTC_NO_PDL");
    on = (e && e[0] && e[0] != '0') ? 0 : 1;
  }
  return on == 1;
}

// Launch with the programmatic-serialization attribute (TTC_NO_PDL=1: without).
template <typename... KArgs, typename... Args>
cudaError_t ttm_launch(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &at;
  cfg.numAttrs = ttm_pdl_on() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

#define TTM_CUDA(call)                                 \
  do {                                                 \
    if ((call) != cudaSuccess) return TT_ERR_CUDA;     \
  } while (0)

// count and scan (and, for the backward, the occurrence lists)
// The batch's bookkeeping: occurrence counts, distinct rows and prefixes,
// their slots and the backward units; with `backward` also the occurrence
// lists.  `reuse`: the counts, slots and units are the lookup's of the same
// batch, still in the workspace, and only the occurrence lists are built
// (from zeroed fill cursors).
tt_status ttm_prepare(int64_t B, const int32_t* idx, const TtmArgs& a, const TtmWs& w, void* ws,
                      bool backward, bool reuse, cudaStream_t st) {
  int gb = (int)std::min<int64_t>((B + 255) / 256, 4 * sm_count());
  if (!reuse) {
    TTM_CUDA(cudaMemsetAsync(at<char>(ws, w.cnt), 0, w.zero_bytes, st));
    int* tsum = at<int>(ws, w.tsum);
    TTM_CUDA(ttm_launch(ttm_count_kernel, gb, 256, 0, st, a, idx));
    TTM_CUDA(ttm_launch(ttm_tile_sum_kernel, w.ntr + w.ntp, kScanThreads, 0, st, a, w.ntr, tsum));
    TTM_CUDA(ttm_launch(ttm_tile_scan_kernel, 1, 1024, 0, st, a, w.ntr, w.ntp, tsum));
    TTM_CUDA(ttm_launch(ttm_tile_write_kernel, w.ntr + w.ntp, kScanThreads, 0, st, a, w.ntr, tsum));
    count_launches(4);
  }
  if (backward) {
    if (reuse) TTM_CUDA(cudaMemsetAsync(a.cursor, 0, (size_t)a.V * sizeof(int), st));
    TTM_CUDA(ttm_launch(ttm_fill_kernel, gb, 256, 0, st, a, idx));
    count_launches(1);
  }
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
  if (desc->flags & ~(TT_ACCUMULATE | TT_REUSE_MERGE)) return TT_ERR_INVALID_ARG;
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
      (int64_t)P.r[2] * P.n[2] > 8192 || pair_rows_smem(P) > 4 * (size_t)kMaxSmemFloats ||
      pair_backward_smem(P) > 4 * (size_t)kMaxSmemFloats)
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
  tt_status s = ttm_prepare(B, idx, a, w, ws, false, false, st);
  if (s != TT_OK) return s;
  ttm_pair_rows_kernel<<<(unsigned)w.pcap, 256, pair_rows_smem(P), st>>>(a);
  ttm_scatter_kernel<<<(unsigned)std::min<int64_t>((B + 7) / 8, 32 * sm_count()), 256, 0, st>>>(
      a, idx, out);
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
  tt_status s = ttm_prepare(B, idx, a, w, ws, true, (P.flags & TT_REUSE_MERGE) != 0, st);
  if (s != TT_OK) return s;
  float* dF1 = dparams + P.core_off[0];
  float* dF2 = dparams + P.core_off[1];
  float* dF3 = P.d == 3 ? dparams + P.core_off[2] : un.sink;
  float* dD1 = dparams + P.diag_off[0];
  float* dD2 = P.d == 3 ? dparams + P.diag_off[1] : un.sink + 32;
  // one thread per float4 column of a row (192 for Dm = 768): no idle lanes
  const int cthreads = (P.Dm % 4 == 0) ? (int)std::min<int64_t>(256, (P.Dm / 4 + 31) / 32 * 32) : 256;
  ttm_chunk_sum_kernel<<<(unsigned)w.unit_cap, cthreads, 0, st>>>(a, dout);
  ttm_pair_backward_kernel<<<(unsigned)w.pcap, 256, pair_backward_smem(P), st>>>(a, dF1, dF2, dF3,
                                                                               dD1, dD2);
  count_launches(2);
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
