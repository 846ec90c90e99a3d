// Merge engine: device side and launcher.  Included once, by tc_fused.cu, so
// that the engine shares the device status word and the operand packing code
// with the tensor-core kernels (one device translation unit).
#pragma once

#include <cstdio>
#include <cstdlib>

#include <vector>

#include "merge_engine.h"

namespace ttc {
namespace {

constexpr int kEngThreads = 512;
constexpr int kEngWarps = kEngThreads / 32;
constexpr int kGK = 512;    // GEMM: K extent staged per pass
constexpr int kGLd = 36;    // GEMM: shared row stride (floats) of a staged [k][m] tile
// GEMM unit dynamic shared memory: A and B tiles, K scales, k-group
// partials, the folded coldot's operand tile and column sums
constexpr int kGemmSmem = 2 * kGK * kGLd + kGK + kEngThreads * 16 + 32 * 32 + 32;
constexpr int kMaxSplits = 32;  // split-K partials of one GEMM task
static_assert(sizeof(EngProgram) <= 30000, "engine program exceeds the kernel parameter limit");
static_assert(kEngThreads == 512, "k-group shifts assume 512 threads");
// Grid barrier: a monotonic 64-bit arrival counter that belongs to one call
// (zeroed in stream order before the launch).  A CTA's own atomicAdd tells it
// which barrier generation it joined, so the target it waits for needs no
// extra read.

// Bounded: false if it timed out (error recorded).  Data produced in one
// phase and read in a later one is read with L2-only loads (__ldcg), so no
// stale L1 line can be observed across a barrier.
__device__ bool eng_grid_barrier(unsigned long long* cnt, unsigned nblocks, int* failed) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    // test hook: the first CTA does not arrive, so the others' waits run out
    const bool skip = blockIdx.x == 0 && debug_take(TT_DEBUG_MERGE_BARRIER);
    if (!skip) {
      const unsigned long long old = atomicAdd(cnt, 1ull);
      const unsigned long long target = (old / nblocks + 1) * nblocks;
      const uint64_t t0 = gtimer();
      const uint64_t limit = *(volatile unsigned long long*)&g_wait_limit_ns;
      while (true) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(cnt) : "memory");
        if (v >= target) break;
        if (gtimer() - t0 > limit) {
          record_error(TT_ERR_TIMEOUT, 100);
          *failed = 1;
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
  return *failed == 0;
}

// Source of element f (flat index into dA (N x rd) or dB (rd x M)) in the
// compacted token sums; null for a pruned rank (the element is 0).
// (32-bit index arithmetic: N*rd and rd*M stay far below 2^31.)
__device__ __forceinline__ const float* eng_gather_src(const EngTask& t, const int* pos,
                                                       int64_t f64) {
  const unsigned f = (unsigned)f64;
  if (t.gather == 1) {
    const unsigned j = f / (unsigned)t.rd;
    const int c = pos[f - j * (unsigned)t.rd];
    return c >= 0 ? t.tc.dAc + (size_t)j * RP + c : nullptr;
  }
  const unsigned a = f / (unsigned)t.M;
  const int c = pos[a];
  return c >= 0 ? t.tc.dBc + (size_t)(f - a * (unsigned)t.M) * RP + c : nullptr;
}

// Asynchronous 4-byte global -> shared copies: a thread issues all of its
// copies without waiting, so a whole staging pass costs one round trip.
__device__ __forceinline__ void cp_async4(float* smem, const float* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(su32(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Issue the copies of one operand tile: element (r, k), r < rows (16 or 32),
// k < kc, of the matrix whose element (r0 + r, k0 + k) is at G[(r0+r)*sr +
// (k0+k)*sk] lands at S[k * kGLd + r]; rows at or past rlim are not
// written.  A warp copies 32-element blocks laid out so that both the global
// reads (unit-stride index fastest) and the shared writes (8 k x 4 rows hit
// 32 distinct banks at row stride 36) are conflict-free.  Every thread keeps
// one row and walks k with a fixed step, so the loop carries no divisions.
// 32-bit offsets: the plan keeps every merge matrix below 2^31 elements.
__device__ __forceinline__ void eng_stage(float* S, int rows, int kc, int r0, int k0, int rlim,
                                          const float* G, int sr, int sk, const EngTask& t,
                                          const int* pos, bool gather) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int rr, kk, step;
  if (sk == 1 && sr != 1) {  // k fastest in memory: blocks of 8 k x 4 rows
    const int lg = rows == 16 ? 2 : 3;  // log2(rows / 4)
    rr = (warp & ((1 << lg) - 1)) * 4 + (lane >> 3);
    kk = (warp >> lg) * 8 + (lane & 7);
    step = (kEngWarps >> lg) * 8;
  } else if (rows == 16) {  // rows fastest: blocks of 16 rows x 2 k
    rr = lane & 15;
    kk = warp * 2 + (lane >> 4);
    step = kEngWarps * 2;
  } else {  // rows fastest: blocks of 32 rows x 1 k
    rr = lane;
    kk = warp;
    step = kEngWarps;
  }
  if (r0 + rr >= rlim) return;
  float* dst = S + kk * kGLd + rr;
  const int dstep = step * kGLd;
  const int f0 = (r0 + rr) * sr + (k0 + kk) * sk;
  const int finc = step * sk;
  if (!gather) {
    const float* src = G + f0;
#pragma unroll 4
    for (; kk < kc; kk += step, dst += dstep, src += finc) cp_async4(dst, src);
    return;
  }
  // gathered operand: f = j * rd + a (dA: row j, compacted column pos[a] of
  // dAc) or f = a * M + o (dB: row o, compacted column pos[a] of dBc); the
  // quotient and remainder by D advance with f
  const bool ga = t.gather == 1;
  const unsigned D = ga ? (unsigned)t.rd : (unsigned)t.M;
  unsigned q = (unsigned)f0 / D, rem = (unsigned)f0 - q * D;
  const unsigned qi = (unsigned)finc / D, ri = (unsigned)finc - qi * D;
  const float* base = ga ? t.tc.dAc : t.tc.dBc;
#pragma unroll 4
  for (; kk < kc; kk += step, dst += dstep) {
    const int c = pos[ga ? rem : q];
    const unsigned row = ga ? q : rem;
    if (c >= 0) cp_async4(dst, base + (size_t)row * RP + c);
    else *dst = 0.f;
    rem += ri;
    q += qi;
    if (rem >= D) {
      rem -= D;
      ++q;
    }
  }
}

// The compaction map of the task's D_d (pos[a]: compacted column of rank a,
// or -1), built when a unit of this CTA first needs it (again when a unit of
// a task with another D_d, another layer, follows): a unit calls it after
// issuing its own copies, so the load of D_d overlaps them.  Uniform across
// the CTA.
__device__ __forceinline__ void ensure_pos(const EngTask& t, int* pos, const float** pos_of) {
  if (*pos_of == t.s) return;  // the map of this task's D_d is the one in pos
  compaction_map(t.s, t.rd, pos, nullptr, nullptr);
  if (threadIdx.x == 0) *pos_of = t.s;
  __syncthreads();
}

// One tm x tn output tile of C over one K split.  The whole K range (in
// passes of kGK) is staged into shared memory with one round of
// asynchronous copies; the kEngThreads threads then split K into
// kEngThreads / (tm*tn/16) groups, each thread owning a 4 x 4 block of the tile, and the group
// partials are summed in a fixed order (deterministic).  Tile counts and
// the split length come from the host; the unit's own index arithmetic is
// 32-bit shifts and masks.
__device__ void eng_gemm_unit(const EngTask& t, int u, int* pos, const float** pos_of, float* dsm,
                              float* rsc, float* csc, int nu) {
  (void)nu;
  TLU_STAMP(nu, 6);
  const GemmArgs& g = t.g;
  const int S = t.splits, TM = t.tm, TN = t.tn;
  const int m = (int)g.m, n = (int)g.n, K = (int)g.k;
  const int tile = (int)(((unsigned long long)(unsigned)u * t.div_s_mul) >> t.div_s_sh);
  const int ks = u - tile * S;
  const int ti = (int)(((unsigned long long)(unsigned)tile * t.div_n_mul) >> t.div_n_sh);
  const int m0 = ti * TM, n0 = (tile - ti * t.tiles_n) * TN;
  const int kb = ks * t.kchunk;
  const int ke = kb + t.kchunk < K ? kb + t.kchunk : K;
  const float* A = static_cast<const float*>(g.A);
  const float* B = static_cast<const float*>(g.B);
  float* As = dsm;
  float* Bs = As + kGK * kGLd;
  float* ksc = Bs + kGK * kGLd;
  float* red = ksc + kGK;
  float* ptile = red + kEngThreads * 16;  // fold: P tile, laid out like red's first group
  float* csum = ptile + 32 * 32;          // fold: column sums of P * v
  const int tid = threadIdx.x;
  const int lgtn4 = TN == 32 ? 3 : 2, lgtn = lgtn4 + 2;
  const int lgG = (TM == 32 ? 3 : 2) + lgtn4;
  const int kg = kEngThreads >> lgG;
  const int grp = tid >> lgG, lid = tid & ((1 << lgG) - 1);
  const int ty = lid >> lgtn4, tx = lid & ((1 << lgtn4) - 1);
  const int mrem = m - m0 < TM ? m - m0 : TM;
  const int nrem = n - n0 < TN ? n - n0 : TN;
  const bool active = ty * 4 < mrem && tx * 4 < nrem;
  const bool gA = t.gather && t.gather_op == 0, gB = t.gather && t.gather_op == 1;
  // epilogue scales of this tile, copied together with the operands
  if (tid < TM) {
    if (g.rscale && tid < mrem) cp_async4(rsc + tid, g.rscale + m0 + tid);
    else rsc[tid] = 1.f;
  }
  if (tid >= 64 && tid < 64 + TN) {
    const int j = tid - 64;
    if (g.cscale && j < nrem) cp_async4(csc + j, g.cscale + (unsigned)(n0 + j) % (unsigned)g.clen);
    else csc[j] = 1.f;
  }
  const bool fold = t.fold_g != nullptr;
  if (fold) {
    for (int o = tid; o < TM * TN; o += kEngThreads) {
      const int i = o >> (TN == 32 ? 5 : 4), j = o & (TN - 1);
      if (i < mrem && j < nrem)
        cp_async4(ptile + o, t.fold_p + (m0 + i) * (int)g.scm + (n0 + j) * (int)g.scn);
    }
    if (tid < TN) csum[tid] = 0.f;
  }
  float acc[4][4] = {};
  for (int k0 = kb; k0 < ke; k0 += kGK) {
    const int kc = ke - k0 < kGK ? ke - k0 : kGK;
    if (k0 != kb) __syncthreads();  // the previous pass's reads are done
    if (k0 == kb) TLU_STAMP(nu, 7);
    // the operand that needs no compaction map goes first
    if (!gA) eng_stage(As, TM, kc, m0, k0, m, A, (int)g.sam, (int)g.sak, t, pos, false);
    if (!gB) eng_stage(Bs, TN, kc, n0, k0, n, B, (int)g.sbn, (int)g.sbk, t, pos, false);
    if (t.gather || t.pack_side) ensure_pos(t, pos, pos_of);
    if (gA) eng_stage(As, TM, kc, m0, k0, m, A, (int)g.sam, (int)g.sak, t, pos, true);
    if (gB) eng_stage(Bs, TN, kc, n0, k0, n, B, (int)g.sbn, (int)g.sbk, t, pos, true);
    if (g.kscale) {
      const unsigned kl = (unsigned)g.klen;
      for (int k = tid; k < kc; k += kEngThreads)
        cp_async4(ksc + k, g.kscale + (unsigned)(k0 + k) % kl);
    }
    if (k0 == kb) TLU_STAMP(nu, 3);
    cp_async_wait_all();
    __syncthreads();
    if (k0 == kb) TLU_STAMP(nu, 4);
    if (active) {
      const int per = (kc + kg - 1) >> (9 - lgG);  // kg = 2^(9 - lgG)
      const int k1 = grp * per;
      const int k2 = k1 + per < kc ? k1 + per : kc;
      const float* ap = As + ty * 4;
      const float* bp = Bs + tx * 4;
#pragma unroll 4
      for (int k = k1; k < k2; ++k) {
        float4 a = *reinterpret_cast<const float4*>(ap + k * kGLd);
        const float4 b = *reinterpret_cast<const float4*>(bp + k * kGLd);
        if (g.kscale) {
          const float sc = ksc[k];
          a.x *= sc; a.y *= sc; a.z *= sc; a.w *= sc;
        }
        const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
    }
  }
  const int tsz = TM * TN;
  if (active) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(red + grp * tsz + (ty * 4 + i) * TN + tx * 4) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
  __syncthreads();
  TLU_STAMP(nu, 5);
  float* C = static_cast<float*>(g.C);
  const int scm = (int)g.scm, scn = (int)g.scn;
  for (int o = tid; o < tsz; o += kEngThreads) {
    const int i = o >> lgtn, j = o & (TN - 1);
    if (i >= mrem || j >= nrem) continue;
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < kEngThreads / 16; ++q)
      if (q < kg) v += red[q * tsz + o];
    const int gm = m0 + i, gn = n0 + j;
    if (fold) {  // last reverse step: the first core's dG and dD, no dQ
      atomicAdd(t.fold_g + gm * scm + gn * scn, v * csc[j]);
      if (csc[j] != 0.f) atomicAdd(&csum[j], ptile[o] * v);
      continue;
    }
    if (S > 1 && g.mode != kAtomic) {
      t.partial[(ks * m + gm) * n + gn] = v;
      continue;
    }
    v *= rsc[i] * csc[j];
    const int ci = gm * scm + gn * scn;
    if (g.mode == kAtomic) {  // each split adds its share into a zeroed C
      atomicAdd(C + ci, v);
      continue;
    }
    C[ci] = g.mode == kAccumulate ? __ldcg(C + ci) + v : v;
    if (t.pack_side) {
      // C is A (N x rd) or B (rd x M), row-major with scm = n, scn = 1
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      const unsigned cu = (unsigned)ci;
      if (t.pack_side == 1) {
        const unsigned jj = cu / (unsigned)t.rd;
        const int c = pos[cu - jj * (unsigned)t.rd];
        if (c >= 0) {
          static_cast<__nv_bfloat16*>(t.tc.Anr)[(size_t)jj * RP + c] = b;
        }
      } else {
        const unsigned a = cu / (unsigned)t.M;
        const int c = pos[a];
        if (c >= 0) {
          const unsigned oo = cu - a * (unsigned)t.M;
          static_cast<__nv_bfloat16*>(t.tc.Bm)[(size_t)c * t.M + oo] = b;
        }
      }
    }
  }
  if (fold) {
    __syncthreads();
    if (tid < nrem && csc[tid] != 0.f) atomicAdd(t.fold_dd + n0 + tid, csum[tid]);
  }
  __syncthreads();  // shared memory is reused by the next unit
}

// kEChain unit: prefixes [p0, p0 + pb) of one side's chain and last-mode
// indices [q0, q0 + sb).  One cooperative pass loads everything the unit
// needs into shared memory (the C_0 rows of its prefixes, the inner cores
// C_1..C_{L-2} whole, the C_{L-1}[:, q0:q0+sb, :] slice and the diagonals),
// so the loads are all in flight together; the chain vectors are then
// rebuilt from shared memory.  P_k rows are written once (by the units with
// q0 == 0), the final rows go to `out` and, on the tensor-core path, to the
// compacted bf16 operands.
constexpr int kChainPB = 32;        // prefixes per unit, unless the phase balancing widens it
constexpr int kChainPBMax = 128;    // the widest unit the balancing makes
constexpr int kChainSmem = 40960;   // floats of dynamic shared memory per CTA
constexpr int kVS = 65;             // shared row stride of the chain vectors (odd: no
                                    // bank conflicts between prefixes)

__host__ __device__ inline int64_t chain_stage_floats(const ChainDesc& c) {
  const int64_t pb = c.pb;
  int64_t f = 2 * pb * kVS + pb * (TT_MAX_D + 1) + pb * TT_MAX_D +
              (int64_t)(c.L > 1 ? c.L - 1 : 0) * 64;
  for (int k = 1; k <= c.L - 2; ++k) f += (int64_t)c.r[k] * c.s[k] * c.r[k + 1];
  f += (int64_t)c.r[c.L - 1] * c.sb * c.r[c.L];
  return f;
}

// Walks e = threadIdx.x, + kEngThreads, ... over a (rows x cols) grid as (r, c)
// with one division up front instead of one per step.
struct Walk2 {
  int r, c, dr, dc, cols;
  __device__ explicit Walk2(int cols_) : cols(cols_) {
    r = (int)threadIdx.x / cols;
    c = (int)threadIdx.x - r * cols;
    dr = kEngThreads / cols;
    dc = kEngThreads - dr * cols;
  }
  __device__ void next() {
    r += dr;
    c += dc;
    if (c >= cols) {
      c -= cols;
      ++r;
    }
  }
};

__device__ void eng_chain_unit(const EngTask& t, int u, int* pos, const float** pos_of,
                               float* dsm, int nu) {
  (void)nu;
  const ChainDesc& c = t.ch;
  const int L = c.L;
  const int pb = c.pb, sb = c.sb;
  const int tid = threadIdx.x;
  const int p0 = (u / c.nsb) * pb;  // prefix counts stay below 2^31
  const int q0 = (u % c.nsb) * sb;
  const int np = (int)(c.nprefix - p0 < pb ? c.nprefix - p0 : pb);
  const int sl = c.s[L - 1], rl1 = c.r[L - 1], rL = c.r[L];
  const int nq = (sl - q0 < sb ? sl - q0 : sb);
  // shared-memory layout
  float* va = dsm;                                              // [pb][kVS] chain vectors
  float* vb = va + pb * kVS;
  int* dig = reinterpret_cast<int*>(vb + pb * kVS);            // [pb][TT_MAX_D + 1] digits, alpha
  int* rowk = dig + pb * (TT_MAX_D + 1);                       // [pb][TT_MAX_D] P_k row of the prefix
  float* dg = reinterpret_cast<float*>(rowk + pb * TT_MAX_D);  // [L-1][64] diagonals
  float* cs[TT_MAX_D] = {};                  // staged inner cores
  float* cur = dg + (L > 1 ? L - 1 : 0) * 64;
  for (int k = 1; k <= L - 2; ++k) {
    cs[k] = cur;
    cur += c.r[k] * c.s[k] * c.r[k + 1];
  }
  float* cf = cur;                           // [rl1][nq][rL] final slice
  // prefix digits and the flat P_k row of each prefix
  for (int pi = tid; pi < np; pi += kEngThreads) {
    unsigned rem = (unsigned)(p0 + pi);
    for (int k = L - 2; k >= 0; --k) {
      const unsigned q = rem / (unsigned)c.s[k];
      dig[pi * (TT_MAX_D + 1) + k] = (int)(rem - q * (unsigned)c.s[k]);
      rem = q;
    }
    dig[pi * (TT_MAX_D + 1) + TT_MAX_D] = (int)rem;  // alpha
    unsigned row = rem;
    for (int k = 0; k <= L - 2; ++k) {
      row = row * (unsigned)c.s[k] + (unsigned)dig[pi * (TT_MAX_D + 1) + k];
      rowk[pi * TT_MAX_D + k] = (int)row;
    }
  }
  __syncthreads();
  // one asynchronous staging pass for everything the unit reads
  const int r1 = c.r[1];
  for (Walk2 w(r1); w.r < np; w.next()) {
    const int* dd = dig + w.r * (TT_MAX_D + 1);
    cp_async4(va + w.r * kVS + w.c, c.core[0] + (dd[TT_MAX_D] * c.s[0] + dd[0]) * r1 + w.c);
  }
  for (int k = 0; k < L - 1; ++k)
    for (int e = tid; e < c.r[k + 1]; e += kEngThreads) cp_async4(dg + k * 64 + e, c.diag[k] + e);
  for (int k = 1; k <= L - 2; ++k) {
    const int n = c.r[k] * c.s[k] * c.r[k + 1];
    for (int e = tid; e < n; e += kEngThreads) cp_async4(cs[k] + e, c.core[k] + e);
  }
  {
    const int w_ = nq * rL;  // one row b of the slice: C_{L-1}[b, q0:q0+nq, :], contiguous
    const float* src = c.core[L - 1] + q0 * rL;
    for (Walk2 w(w_); w.r < rl1; w.next()) cp_async4(cf + w.r * w_ + w.c, src + w.r * sl * rL + w.c);
  }
  if (t.pack_side) ensure_pos(t, pos, pos_of);
  cp_async_wait_all();
  __syncthreads();
  TLU_STAMP(nu, 3);
  // the chain vectors carry the diagonal that follows them: v <- v * E_0
  for (Walk2 w(r1); w.r < np; w.next()) va[w.r * kVS + w.c] *= dg[w.c];
  __syncthreads();
  TLU_STAMP(nu, 4);
  // steps 1 .. L-2: v <- v . C_k[:, d_k, :] (then times E_k); lanes walk
  // the columns, so the P_k rows are written coalesced
  for (int k = 1; k <= L - 2; ++k) {
    const int rk = c.r[k], rk1 = c.r[k + 1], sk = c.s[k];
    const float* Ek = dg + k * 64;
    const int bstride = sk * rk1;
    float* prow = (q0 == 0) ? c.prow[k] : nullptr;
    for (Walk2 w(rk1); w.r < np; w.next()) {
      const int pi = w.r, col = w.c;
      const float* Ck = cs[k] + dig[pi * (TT_MAX_D + 1) + k] * rk1 + col;
      const float* v = va + pi * kVS;
      float a0 = 0.f, a1 = 0.f;
      int b = 0;
      for (; b + 1 < rk; b += 2) {
        a0 = fmaf(v[b], Ck[b * bstride], a0);
        a1 = fmaf(v[b + 1], Ck[(b + 1) * bstride], a1);
      }
      if (b < rk) a0 = fmaf(v[b], Ck[b * bstride], a0);
      const float acc = a0 + a1;
      vb[pi * kVS + col] = acc * Ek[col];
      if (prow) prow[rowk[pi * TT_MAX_D + k] * rk1 + col] = acc;
    }
    __syncthreads();
    float* tmp = va;
    va = vb;
    vb = tmp;
  }
  TLU_STAMP(nu, 5);
  // final rows (prefix, q) = v . C_{L-1}[:, q, :].  Item (prefix group of
  // four, z = q * rL + col): lanes walk z, along which both the staged slice
  // and the output rows are contiguous, so the stores coalesce
  const int zw = nq * rL;
  const int npg = (np + 3) >> 2;
  for (Walk2 w(zw); w.r < npg; w.next()) {
    const int pi0 = w.r * 4, z = w.c;
    const int npi = np - pi0 < 4 ? np - pi0 : 4;
    const float* Cz = cf + z;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int b = 0; b < rl1; ++b) {
      const float y = Cz[b * zw];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (i < npi) acc[i] = fmaf(va[(pi0 + i) * kVS + b], y, acc[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (i >= npi) break;
      const float v = acc[i];
      const int f = ((p0 + pi0 + i) * sl + q0) * rL + z;  // flat index into P_{L-1}
      if (c.out) c.out[f] = v;
      if (!t.pack_side) continue;
      const __nv_bfloat16 bv = __float2bfloat16_rn(v);
      if (t.pack_side == 1) {  // A (N x rd): f = j * rd + a
        const unsigned jj = (unsigned)f / (unsigned)t.rd;
        const int cc = pos[(unsigned)f - jj * (unsigned)t.rd];
        if (cc >= 0) static_cast<__nv_bfloat16*>(t.tc.Anr)[(size_t)jj * RP + cc] = bv;
      } else {  // B (rd x M): f = a * M + o
        const unsigned a = (unsigned)f / (unsigned)t.M;
        const int cc = pos[a];
        if (cc >= 0) {
          const unsigned o = (unsigned)f - a * (unsigned)t.M;
          static_cast<__nv_bfloat16*>(t.tc.Bm)[(size_t)cc * t.M + o] = bv;
        }
      }
    }
  }
  __syncthreads();
}

__device__ void eng_gemm_final_unit(const EngTask& t, int u) {
  const GemmArgs& g = t.g;
  const int64_t i = (int64_t)u * kEngThreads + threadIdx.x;
  if (i >= g.m * g.n) return;
  const unsigned gm = (unsigned)i / (unsigned)g.n, gn = (unsigned)i - gm * (unsigned)g.n;
  // all of the split partials in flight at once, summed in split order
  float pv[kMaxSplits];
#pragma unroll
  for (int ks = 0; ks < kMaxSplits; ++ks)
    pv[ks] = ks < t.splits ? __ldcg(t.partial + (int64_t)ks * g.m * g.n + i) : 0.f;
  float v = 0.f;
#pragma unroll
  for (int ks = 0; ks < kMaxSplits; ++ks) v += pv[ks];
  if (g.rscale) v *= g.rscale[gm];
  if (g.cscale) v *= g.cscale[gn % (unsigned)g.clen];
  float* C = static_cast<float*>(g.C);
  const int64_t ci = gm * g.scm + gn * g.scn;
  C[ci] = g.mode == kAccumulate ? __ldcg(C + ci) + v : v;
}

__device__ void eng_coldot_unit(const EngTask& t, int c, float* red) {
  float s = 0.f;
#pragma unroll 8
  for (int64_t u = threadIdx.x; u < t.n; u += blockDim.x)
    s += __ldcg(t.x + u * t.sx + c) * __ldcg(t.y + u * t.sy + c);
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    s = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) {
      const bool keep = !t.s || t.s[c] != 0.f;
      if (t.acc) {
        if (keep) t.out[c] += s;
      } else {
        t.out[c] = keep ? s : 0.f;
      }
    }
  }
  __syncthreads();
}

__device__ void eng_scale_unit(const EngTask& t, int u) {
  const int64_t base = (int64_t)u * t.chunk;
  for (int e = threadIdx.x; e < t.chunk; e += blockDim.x) {
    const int64_t i = base + e;
    if (i >= t.n) break;
    float v = t.x ? __ldcg(t.x + i) : 0.f;
    if (t.s) v *= t.s[(unsigned)i % (unsigned)t.len];
    t.out[i] = t.acc ? __ldcg(t.out + i) + v : v;
  }
}

__device__ void eng_rank_unit(const EngTask& t, int u) {
  const int64_t base = (int64_t)u * t.chunk;
  for (int e = threadIdx.x; e < t.chunk; e += blockDim.x) {
    const int64_t i = base + e;
    if (i >= t.n) break;
    rank_step_elem(t.out, t.dA, (int)i, i < t.len, t.rk);
  }
}

constexpr int kEngSmem = kGemmSmem > kChainSmem ? kGemmSmem : kChainSmem;

__global__ void __launch_bounds__(kEngThreads) eng_kernel(const __grid_constant__ EngProgram prog) {
  extern __shared__ __align__(16) float eng_dsm[];  // kEngSmem floats: GEMM or chain staging
  __shared__ float red[32];
  __shared__ int pos[RP];
  __shared__ float rsc[32], csc[32];
  // Tasks are read straight from the parameter space: every thread of a warp
  // reads the same field, which the constant cache broadcasts.  (Copying
  // the whole program to shared memory first costs several microseconds:
  // per-lane addresses into parameter space serialise.)
  const EngProgram& p = prog;
  __shared__ int failed;
  pdl_wait();  // params and workspace may be written by the previous grid
  pdl_trigger();
  if (threadIdx.x == 0) {
    failed = 0;
    TL_STAMP(p.nphases == 1 ? 2 : 3, 0);
  }
  __shared__ const float* pos_of;  // the D_d whose compaction map pos holds
  if (threadIdx.x == 0) pos_of = nullptr;
  __syncthreads();
#ifdef TTC_TIMELINE
  int nu = 0;
#else
  constexpr int nu = 0;
#endif
  for (int ph = 0; ph < p.nphases; ++ph) {
    const int t0 = p.phase_begin[ph], t1 = p.phase_begin[ph + 1];
    const int total = p.ptotal[ph];
    // Units are dealt in waves of gridDim.x, costliest tasks first, and every
    // other wave in reverse CTA order, so that the CTAs with the cheapest
    // unit of one wave take the costliest of the next.
    for (int w = 0; w * (int)gridDim.x < total; ++w) {
      const int u = w * (int)gridDim.x +
                    ((w & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
      if (u >= total) continue;
      int o = t0;
      while (o + 1 < t1 && u >= p.ustart[o + 1]) ++o;
      const int uu = u - p.ustart[o];
      const int t = p.order[o];
      const EngTask& k = p.t[t];
#ifdef TTC_TIMELINE
      if (threadIdx.x == 0 && nu < 8) {
        g_tlu[blockIdx.x & 255][nu][0] = ph * 100 + t;
        g_tlu[blockIdx.x & 255][nu][1] = gtimer();
      }
#endif
      switch (k.kind) {
        case kEGemm: eng_gemm_unit(k, uu, pos, &pos_of, eng_dsm, rsc, csc, nu); break;
        case kEGemmFinal: eng_gemm_final_unit(k, uu); break;
        case kEColdot: eng_coldot_unit(k, uu, red); break;
        case kEScale: eng_scale_unit(k, uu); break;
        case kEPack:
          tc_pack_unit(k.A, k.B, k.s, k.rd, k.N, k.M, k.tc, k.zero, k.pad_only, k.chunk, uu);
          break;
        case kEDd:
          tc_dd_unit(k.tc, k.s, k.rd, k.out, k.acc);
          break;
        case kEChain: eng_chain_unit(k, uu, pos, &pos_of, eng_dsm, nu); break;
        case kERank: eng_rank_unit(k, uu); break;
        case kEUnpack:
          tc_unpack_unit(k.tc, k.s, k.rd, k.N, k.M, k.dA, k.dB, k.out, k.acc, k.chunk, uu);
          break;
        default: break;
      }
#ifdef TTC_TIMELINE
      __syncthreads();
      if (threadIdx.x == 0 && nu < 8) g_tlu[blockIdx.x & 255][nu][2] = gtimer();
      ++nu;
#endif
    }
    if (threadIdx.x == 0) TL_STAMP(p.nphases == 1 ? 2 : 3, 1 + 2 * ph);
    if (ph + 1 < p.nphases && !eng_grid_barrier(p.bar, gridDim.x, &failed)) return;
    if (threadIdx.x == 0) TL_STAMP(p.nphases == 1 ? 2 : 3, 2 + 2 * ph);
  }
}

}  // namespace

// ---- host side -------------------------------------------------------------

int eng_sm_count() { return device_sms(); }

void EngBuilder::begin_phase() {
  if (p.nphases > 0) balance(eng_sm_count());
  if (p.nphases >= kEngMaxPhases) {
    overflow = true;
    return;
  }
  p.phase_begin[p.nphases++] = p.ntasks;
}

EngTask* EngBuilder::add() {
  static EngTask dummy;
  if (p.ntasks >= kEngMaxTasks || p.nphases == 0) {
    overflow = true;
    return &dummy;
  }
  p.t[p.ntasks] = EngTask();
  return &p.t[p.ntasks++];
}

void EngBuilder::end() {
  if (p.nphases > 0) balance(eng_sm_count());
  p.phase_begin[p.nphases] = p.ntasks;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t eng_partial_floats(int64_t m, int64_t n, int64_t k) {
  (void)k;
  // splits happen only below 128 tiles of at most 32 x 32, with at most
  // ceil(128 / tiles) splits: splits * m * n < 2 * 128 * 1024
  const size_t full = (size_t)(m * n) * kMaxSplits;
  const size_t bound = (size_t)2 * 128 * 1024;
  return full < bound ? full : bound;
}

// x / d for 0 <= x < 2^31 as (x * mul) >> sh: with l = ceil(log2 d) and
// mul = ceil(2^(31+l) / d), x * mul / 2^(31+l) exceeds x / d by less than
// 2^31 / 2^(31+l) <= 1 / d, which never reaches the next integer.
static void eng_divisor(int d, unsigned long long* mul, int* sh) {
  int l = 0;
  while ((1ll << l) < d) ++l;
  const unsigned long long num = 1ull << (31 + l);
  *mul = (num + (unsigned long long)d - 1) / (unsigned long long)d;
  *sh = 31 + l;
}

// Sets a GEMM task's tile (tm x tn) and split count, and what follows.
static void eng_gemm_set(EngTask* t, int tm, int tn, int splits) {
  const GemmArgs& g = t->g;
  t->tm = tm;
  t->tn = tn;
  t->splits = splits;
  t->units = (int)(ceil_div(g.m, tm) * ceil_div(g.n, tn) * splits);
  t->tiles_n = (int)ceil_div(g.n, tn);
  t->kchunk = (int)ceil_div(g.k, splits);
  eng_divisor(t->splits, &t->div_s_mul, &t->div_s_sh);
  eng_divisor(t->tiles_n, &t->div_n_mul, &t->div_n_sh);
}

// Tile (16 or 32 a side) and split choice: the configuration with the most
// units not above max_units (ties: larger tiles, then fewer splits); if none
// fits, the one with the fewest units.  A split keeps >= 48 of K.
static void eng_gemm_config(EngTask* t, int max_units) {
  const GemmArgs& g = t->g;
  const bool atomic = t->atomic_splits && g.mode == kAtomic;
  const bool can_split = atomic || t->partial != nullptr;
  int64_t maxs = can_split ? ceil_div(g.k, 48) : 1;
  if (maxs > kMaxSplits) maxs = kMaxSplits;
  if (maxs < 1) maxs = 1;
  int64_t fit_u = -1, min_u = -1;
  int fit[3] = {32, 32, 1}, mn[3] = {32, 32, 1};
  for (int tm : {32, 16}) {
    if (tm == 32 && g.m <= 16) continue;
    for (int tn : {32, 16}) {
      if (tn == 32 && g.n <= 16) continue;
      const int64_t tiles = ceil_div(g.m, tm) * ceil_div(g.n, tn);
      for (int64_t s = 1; s <= maxs; ++s) {
        if (s > 1 && !atomic && s * g.m * g.n > t->pcap) break;
        const int64_t u = tiles * s;
        if (u <= max_units && (u > fit_u || (u == fit_u && tm * tn > fit[0] * fit[1]))) {
          fit_u = u;
          fit[0] = tm; fit[1] = tn; fit[2] = (int)s;
        }
        if (min_u < 0 || u < min_u || (u == min_u && tm * tn > mn[0] * mn[1])) {
          min_u = u;
          mn[0] = tm; mn[1] = tn; mn[2] = (int)s;
        }
      }
    }
  }
  const int* c = fit_u >= 0 ? fit : mn;
  eng_gemm_set(t, c[0], c[1], c[2]);
}

// Every configuration eng_gemm_config may choose for t (at most
// kEngMaxConfigs): tile, splits, units and unit cost.
struct EngCfg {
  int tm, tn, splits, units;
  double cost;
};
constexpr int kEngMaxConfigs = 4 * kMaxSplits;
static double eng_unit_cost(const EngTask& k);
static int eng_gemm_configs(const EngTask& t, EngCfg* out) {
  const GemmArgs& g = t.g;
  const bool atomic = t.atomic_splits && g.mode == kAtomic;
  const bool can_split = atomic || t.partial != nullptr;
  int64_t maxs = can_split ? ceil_div(g.k, 48) : 1;
  if (maxs > kMaxSplits) maxs = kMaxSplits;
  if (maxs < 1) maxs = 1;
  int n = 0;
  EngTask tmp = t;
  for (int tm : {32, 16}) {
    if (tm == 32 && g.m <= 16) continue;
    for (int tn : {32, 16}) {
      if (tn == 32 && g.n <= 16) continue;
      for (int64_t sp = 1; sp <= maxs && n < kEngMaxConfigs; ++sp) {
        if (sp > 1 && !atomic && sp * g.m * g.n > t.pcap) break;
        eng_gemm_set(&tmp, tm, tn, (int)sp);
        out[n++] = {tm, tn, (int)sp, tmp.units, eng_unit_cost(tmp)};
      }
    }
  }
  return n;
}

void eng_gemm_task(EngTask* t, const GemmArgs& g, float* partial_ws, size_t partial_cap,
                   bool atomic_splits, int max_units) {
  t->kind = kEGemm;
  t->g = g;
  t->atomic_splits = atomic_splits ? 1 : 0;
  // split-K partials (for a final task in a later phase) unless the splits
  // add atomically; the device reads `partial` only when splits > 1
  t->partial = (atomic_splits && g.mode == kAtomic) ? nullptr : partial_ws;
  t->pcap = t->partial ? (int64_t)partial_cap : 0;
  eng_gemm_config(t, max_units);
}

// Rough cost of one unit of a task (about nanoseconds: for ordering the units
// and for the balancing's cap): a GEMM unit pays a staging round trip plus
// its tile's K extent; a chain unit stages whole cores.
static double eng_unit_cost(const EngTask& k) {
  switch (k.kind) {
    case kEGemm:
      // a gathered operand (token sums through the compaction map) stages
      // element by element from rows 64 floats apart: about twice the cost
      // a float of a contiguous one
      return 2000.0 + 0.25 * (double)k.kchunk * (k.tm + k.tn) + (k.fold_g ? 500.0 : 0.0) +
             (k.gather || k.pack_side ? 500.0 : 0.0) +
             (k.gather ? 0.5 * (double)k.kchunk * (k.gather_op == 0 ? k.tm : k.tn) : 0.0);
    case kEChain: return 6000.0;
    case kEGemmFinal: return 400.0 + 50.0 * k.splits;
    case kEColdot: return 800.0 + 0.5 * (double)k.n;  // one column over n strided rows
    case kEPack:
    case kEUnpack:
    case kEDd: return 800.0;
    default: return 400.0;
  }
}

// One step wider for a task whose units are latency-bound: a chain task
// takes twice the prefixes a unit (while its staging fits the shared memory),
// a pack or unpack task twice the elements.  False when the task can not
// widen or its unit count would not drop.
static bool eng_widen(EngTask* t) {
  if (t->kind == kEChain) {
    ChainDesc c = t->ch;
    if (2 * c.pb > kChainPBMax || c.pb >= c.nprefix) return false;
    c.pb *= 2;
    if (chain_stage_floats(c) > kChainSmem) return false;
    const int units = (int)(ceil_div(c.nprefix, c.pb) * c.nsb);
    if (units >= t->units) return false;
    t->ch = c;
    t->units = units;
    return true;
  }
  if (t->kind == kEPack || t->kind == kEUnpack) {
    if (2 * t->chunk > kPackPerMax) return false;
    const int w = t->kind == kEPack ? RP : t->rd;
    const int64_t n = ((int64_t)t->N + t->M) * w + w;
    const int units = (int)ceil_div(n, 2 * t->chunk);
    if (units >= t->units) return false;
    t->chunk *= 2;
    t->units = units;
    return true;
  }
  return false;
}

// The phase's units in as few waves of `budget` CTAs as the task shapes allow:
// GEMM tasks re-tiled; chain, pack and unpack tasks widened (their units are
// latency-bound, so fewer waves of somewhat longer units finish sooner).  A
// GEMM is not re-tiled into units longer (by the cost model) than the
// phase's longest unit that nothing can shorten, and at least 8 us: one long
// unit (a whole K of 1024 on one CTA) would outlast the waves it saves.
void EngBuilder::balance(int budget) {
  const int t0 = p.phase_begin[p.nphases - 1];
  double cap = 8000.0;
  bool frozen[kEngMaxTasks] = {};
  for (int i = t0; i < p.ntasks; ++i)
    if (p.t[i].kind != kEGemm && eng_unit_cost(p.t[i]) > cap) cap = eng_unit_cost(p.t[i]);
  // aim at the fewest waves that the narrowest configuration allows
  int64_t min_total = 0;
  for (int i = t0; i < p.ntasks; ++i) {
    EngTask probe = p.t[i];
    if (probe.kind == kEGemm) eng_gemm_config(&probe, 0);
    while (eng_widen(&probe)) {
    }
    min_total += probe.units;
  }
  if (budget < 1) budget = 1;
  const bool one_wave = min_total <= budget;
  if (min_total > budget) budget = (int)(ceil_div(min_total, budget) * budget);
  for (int iter = 0; iter < 256; ++iter) {
    int64_t total = 0;
    for (int i = t0; i < p.ntasks; ++i) total += p.t[i].units;
    if (total <= budget) break;
    // shrink the task with the most units that can still shrink
    int best = -1;
    for (int i = t0; i < p.ntasks; ++i) {
      EngTask& k = p.t[i];
      if (frozen[i] || (best >= 0 && k.units <= p.t[best].units)) continue;
      EngTask probe = k;
      bool can = false;
      if (k.kind == kEGemm) {
        eng_gemm_config(&probe, 0);  // fewest units
        can = probe.units < k.units;
      } else {
        can = eng_widen(&probe);
      }
      if (can) best = i;
    }
    if (best < 0) break;
    EngTask& k = p.t[best];
    if (k.kind == kEGemm) {
      const EngTask before = k;
      const int64_t want = k.units - (total - budget);
      eng_gemm_config(&k, (int)(want > 0 ? want : 0));
      if (eng_unit_cost(k) > cap && eng_unit_cost(k) > eng_unit_cost(before)) {
        // the fewest units whose cost stays under the cap, then no further
        k = before;
        for (int w = (int)(want > 0 ? want : 0) + 1; w < before.units; ++w) {
          EngTask probe = before;
          eng_gemm_config(&probe, w);
          if (probe.units < before.units && eng_unit_cost(probe) <= cap) {
            k = probe;
            break;
          }
        }
        frozen[best] = true;
      }
    } else {
      eng_widen(&k);
    }
  }
  if (one_wave) refine(budget);
  else refine_waves();
}

// The phase's length as eng_kernel deals it: tasks costliest unit first,
// waves of `grid` units, every other wave in reverse CTA order; the largest
// sum of unit costs a CTA gets.
static double eng_phase_makespan(const EngProgram& p, int t0, int t1, int grid) {
  int order[kEngMaxTasks];
  int n = 0;
  for (int i = t0; i < t1; ++i) {
    const double c = eng_unit_cost(p.t[i]);
    int j = n;
    for (; j > 0 && eng_unit_cost(p.t[order[j - 1]]) < c; --j) order[j] = order[j - 1];
    order[j] = i;
    ++n;
  }
  std::vector<double> load((size_t)grid, 0.0);
  int64_t u = 0;
  for (int o = 0; o < n; ++o) {
    const EngTask& k = p.t[order[o]];
    const double c = eng_unit_cost(k);
    for (int i = 0; i < k.units; ++i, ++u) {
      const int64_t w = u / grid, r = u - w * grid;
      load[(size_t)((w & 1) ? grid - 1 - r : r)] += c;
    }
  }
  double m = 0.0;
  for (double v : load) m = v > m ? v : m;
  return m;
}

// A phase of several waves: GEMM tasks take the configuration (tile and K
// splits) that shortens the dealt phase the most, one task at a time, while
// any step shortens it.  Host work only: the candidate configurations of a
// task are those within a factor four of its units.
void EngBuilder::refine_waves() {
  const int t0 = p.phase_begin[p.nphases - 1], t1 = p.ntasks;
  const int grid = eng_sm_count();
  EngCfg cfg[kEngMaxConfigs];
  double best = eng_phase_makespan(p, t0, t1, grid);
  for (int iter = 0; iter < 8; ++iter) {
    bool improved = false;
    for (int i = t0; i < t1; ++i) {
      if (p.t[i].kind != kEGemm) continue;
      const EngTask keep = p.t[i];
      const int nc = eng_gemm_configs(keep, cfg);
      int pick = -1;
      for (int c = 0; c < nc; ++c) {
        if (cfg[c].units == keep.units && cfg[c].tm == keep.tm && cfg[c].tn == keep.tn) continue;
        if (cfg[c].units > 4 * keep.units || 4 * cfg[c].units < keep.units) continue;
        eng_gemm_set(&p.t[i], cfg[c].tm, cfg[c].tn, cfg[c].splits);
        const double m = eng_phase_makespan(p, t0, t1, grid);
        if (m < best - 1.0) {
          best = m;
          pick = c;
        }
      }
      p.t[i] = keep;
      if (pick >= 0) {
        eng_gemm_set(&p.t[i], cfg[pick].tm, cfg[pick].tn, cfg[pick].splits);
        improved = true;
      }
    }
    if (!improved) return;
  }
}

// In a phase of one unit a CTA the phase lasts as long as its costliest
// unit: while that unit is a GEMM's, give that task a finer configuration
// (more units, each cheaper) if the phase still fits `budget` units, making
// room where needed by coarsening other GEMM tasks as far as their units stay
// below the new maximum.  Stops when no step lowers the maximum.
void EngBuilder::refine(int budget) {
  const int t0 = p.phase_begin[p.nphases - 1];
  std::vector<EngCfg> cfgs((size_t)(p.ntasks - t0) * kEngMaxConfigs);
  std::vector<int> ncfg((size_t)(p.ntasks - t0));
  for (int iter = 0; iter < 16; ++iter) {
    int64_t total = 0;
    int hi = -1;
    for (int i = t0; i < p.ntasks; ++i) {
      total += p.t[i].units;
      if (hi < 0 || eng_unit_cost(p.t[i]) > eng_unit_cost(p.t[hi])) hi = i;
    }
    if (hi < 0 || p.t[hi].kind != kEGemm || total > budget) return;
    const double cmax = eng_unit_cost(p.t[hi]);
    double others = 0.0;  // the costliest unit of every other task
    for (int i = t0; i < p.ntasks; ++i)
      if (i != hi && eng_unit_cost(p.t[i]) > others) others = eng_unit_cost(p.t[i]);
    for (int i = t0; i < p.ntasks; ++i)
      ncfg[i - t0] = p.t[i].kind == kEGemm
                         ? eng_gemm_configs(p.t[i], &cfgs[(size_t)(i - t0) * kEngMaxConfigs])
                         : 0;
    const EngCfg* cfg = &cfgs[(size_t)(hi - t0) * kEngMaxConfigs];
    double best_max = cmax;
    int best_c = -1;
    int best_sub[kEngMaxTasks];  // per other task its new configuration (-1: unchanged)
    for (int c = 0; c < ncfg[hi - t0]; ++c) {
      if (cfg[c].units <= p.t[hi].units) continue;
      const double newmax = cfg[c].cost > others ? cfg[c].cost : others;
      if (newmax >= best_max) continue;
      // units to free elsewhere: the GEMM tasks coarsened to their fewest
      // units whose cost stays at or below newmax
      int64_t need = total - p.t[hi].units + cfg[c].units - budget;
      int sub[kEngMaxTasks];
      for (int i = t0; i < p.ntasks; ++i) sub[i] = -1;
      for (int i = t0; i < p.ntasks && need > 0; ++i) {
        if (i == hi) continue;
        const EngCfg* alt = &cfgs[(size_t)(i - t0) * kEngMaxConfigs];
        int pick = -1;
        for (int a2 = 0; a2 < ncfg[i - t0]; ++a2)
          if (alt[a2].units < p.t[i].units && alt[a2].cost <= newmax &&
              (pick < 0 || alt[a2].units < alt[pick].units))
            pick = a2;
        if (pick >= 0) {
          need -= p.t[i].units - alt[pick].units;
          sub[i] = pick;
        }
      }
      if (need > 0) continue;
      best_max = newmax;
      best_c = c;
      for (int i = t0; i < p.ntasks; ++i) best_sub[i] = sub[i];
    }
    if (best_c < 0) return;
    const EngCfg h = cfg[best_c];
    for (int i = t0; i < p.ntasks; ++i)
      if (best_sub[i] >= 0) {
        const EngCfg& a2 = cfgs[(size_t)(i - t0) * kEngMaxConfigs + best_sub[i]];
        eng_gemm_set(&p.t[i], a2.tm, a2.tn, a2.splits);
      }
    eng_gemm_set(&p.t[hi], h.tm, h.tn, h.splits);
  }
}

void eng_dd_task(EngTask* t, const LayerPlan& L, const TcPtrs& tc, const float* Dmid,
                 float* dDout, bool acc) {
  t->kind = kEDd;
  t->s = Dmid;
  t->tc = tc;
  t->rd = L.rd;
  t->out = dDout;
  t->acc = acc ? 1 : 0;
  t->units = 1;
}

void eng_pack_task(EngTask* t, const LayerPlan& L, const float* A, const float* B,
                   const float* Dmid, const TcPtrs& tc, bool zero_grads, bool pad_only) {
  t->kind = kEPack;
  t->pad_only = pad_only ? 1 : 0;
  t->A = A;
  t->B = B;
  t->s = Dmid;
  t->rd = L.rd;
  t->N = (int)L.N;
  t->M = (int)L.M;
  t->tc = tc;
  t->zero = zero_grads ? 1 : 0;
  t->chunk = kPackPer;
  t->units = (int)ceil_div((L.N + L.M) * RP + RP, t->chunk);
}

void eng_unpack_task(EngTask* t, const LayerPlan& L, const TcPtrs& tc, const float* Dmid,
                     float* dA, float* dB, float* dDout, bool acc) {
  t->kind = kEUnpack;
  t->s = Dmid;
  t->tc = tc;
  t->rd = L.rd;
  t->N = (int)L.N;
  t->M = (int)L.M;
  t->dA = dA;
  t->dB = dB;
  t->out = dDout;
  t->acc = acc ? 1 : 0;
  t->chunk = kPackPer;
  t->units = (int)ceil_div((L.N + L.M) * L.rd + L.rd, t->chunk);
}

void eng_rank_task(EngTask* t, const LayerPlan& L, float* params, float* dparams,
                   const RankStep& r) {
  t->kind = kERank;
  t->out = params;
  t->dA = dparams;
  t->n = (int64_t)L.n_floats;
  t->len = (int)L.diag_off[0];  // the cores come first
  t->rk = r;
  t->chunk = 4096;
  t->units = (int)ceil_div(t->n, t->chunk);
}

bool eng_chain_task(EngTask* t, const ChainDesc& c) {
  t->kind = kEChain;
  t->ch = c;
  // split the last mode when the last core is large, so that a unit stages
  // only a slice of it
  const int64_t last = (int64_t)c.r[c.L - 1] * c.s[c.L - 1] * c.r[c.L];
  t->ch.sb = last > 4096 ? 1 : c.s[c.L - 1];
  t->ch.nsb = (c.s[c.L - 1] + t->ch.sb - 1) / t->ch.sb;
  t->ch.pb = kChainPB;
  t->units = (int)(ceil_div(c.nprefix, kChainPB) * t->ch.nsb);
  for (int k = 0; k <= c.L; ++k)
    if (c.r[k] > 64) return false;
  return chain_stage_floats(t->ch) <= kChainSmem;
}

void eng_gemm_final_task(EngTask* t, const EngTask& gemm) {
  t->kind = kEGemmFinal;
  t->g = gemm.g;
  t->splits = gemm.splits;
  t->partial = gemm.partial;
  t->units = (int)ceil_div(gemm.g.m * gemm.g.n, kEngThreads);
}

static void eng_dump(const EngProgram& p) {
  for (int ph = 0; ph < p.nphases; ++ph) {
    fprintf(stderr, "engine phase %d\n", ph);
    for (int o = p.phase_begin[ph]; o < p.phase_begin[ph + 1]; ++o) {
      const EngTask& k = p.t[p.order[o]];
      fprintf(stderr,
              "  task %2d kind %d units %4d  m %lld n %lld k %lld  tile %dx%d splits %d kchunk %d"
              "%s%s%s\n",
              (int)p.order[o], k.kind, k.units, (long long)k.g.m, (long long)k.g.n,
              (long long)k.g.k, k.tm, k.tn, k.splits, k.kchunk, k.fold_g ? " fold" : "",
              k.gather ? " gather" : "", k.pack_side ? " pack" : "");
    }
  }
}

cudaError_t eng_launch(const EngProgram& prog, cudaStream_t st) {
  // the shared-memory opt-in and the occupancy check, once per device
  static PerDevice setup;
  cudaError_t se = setup.get([] {
    int per = 0;
    cudaError_t e = cudaFuncSetAttribute(eng_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kEngSmem * sizeof(float)));
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, eng_kernel, kEngThreads,
                                                        kEngSmem * sizeof(float));
    return e != cudaSuccess ? e : per > 0 ? cudaSuccess : cudaErrorLaunchFailure;
  });
  if (se != cudaSuccess) return se;
  const int grid = device_sms();
  if (prog.nphases > 1 && !prog.bar) return cudaErrorInvalidValue;
  EngProgram p = prog;
  for (int ph = 0; ph < p.nphases; ++ph) {  // costliest units first, stable
    const int a = p.phase_begin[ph], b = p.phase_begin[ph + 1];
    for (int i = a; i < b; ++i) p.order[i] = (unsigned char)i;
    for (int i = a + 1; i < b; ++i) {
      const unsigned char v = p.order[i];
      const double cv = eng_unit_cost(p.t[v]);
      int j = i;
      for (; j > a && eng_unit_cost(p.t[p.order[j - 1]]) < cv; --j) p.order[j] = p.order[j - 1];
      p.order[j] = v;
    }
    int acc = 0;
    for (int i = a; i < b; ++i) {
      p.ustart[i] = acc;
      acc += p.t[p.order[i]].units;
    }
    p.ptotal[ph] = acc;
  }
  static int dumps = 0;
  if (getenv("TTC_ENG_DUMP") && dumps < 4) {
    ++dumps;
    eng_dump(p);
  }
  int g = grid;
  // Only a grid barrier needs every CTA resident at once: a one-phase
  // program launches as an ordinary grid, whose CTAs start as the previous
  // grid's CTAs leave their SMs (with programmatic launch, before it ends).
  bool coop = p.nphases > 1;
#ifdef TTC_TIMELINE
  // measurement builds only: grid size and launch kind from the environment
  if (const char* e = getenv("TTC_ENG_GRID")) g = atoi(e) > 0 && atoi(e) < grid ? atoi(e) : grid;
  if (getenv("TTC_ENG_NONCOOP")) coop = false;
#endif
  cudaError_t e = launch_ex(eng_kernel, dim3(g), dim3(kEngThreads), kEngSmem * sizeof(float), st,
                            coop, p);
  count_launches(1);
  return e;
}

}  // namespace ttc
