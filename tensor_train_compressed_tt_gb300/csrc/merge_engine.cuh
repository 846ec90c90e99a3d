// Merge engine: device side and launcher.  Included once, by tc_fused.cu, so
// that the engine shares the device status word and the operand packing code
// with the tensor-core kernels (one device translation unit).
#pragma once

#include <atomic>

#include "merge_engine.h"

namespace ttc {
namespace {

constexpr int kEngThreads = 256;
constexpr int kET = 32;   // GEMM tile (kET x kET outputs per unit)
constexpr int kEK = 128;  // K slice staged per iteration (all loads in flight at once)
constexpr int kBarSlots = 64;
static_assert(sizeof(EngProgram) <= 30000, "engine program exceeds the kernel parameter limit");
static_assert(sizeof(EngProgram) % 16 == 0, "the program is copied in 16-byte pieces");

// Grid barrier: one monotonic 64-bit arrival counter per slot (own
// 128-byte line).  A CTA's own atomicAdd tells it which barrier generation
// it joined, so the target it waits for needs no extra read and the counter
// never has to be reset: every launch on a slot uses the same grid size and
// launches on one slot are serialised by their stream.
struct EngBarSlot {
  unsigned long long count;
  unsigned long long pad[15];
};
__device__ EngBarSlot g_eng_bar[kBarSlots];

// Bounded: false if it timed out (error recorded).  Data produced in one
// phase and read in a later one is read with L2-only loads (__ldcg), so no
// stale L1 line can be observed across a barrier.
__device__ bool eng_grid_barrier(unsigned slot, unsigned nblocks, int* failed) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long* cnt = &g_eng_bar[slot].count;
    __threadfence();
    const unsigned long long old = atomicAdd(cnt, 1ull);
    const unsigned long long target = (old / nblocks + 1) * nblocks;
    const uint64_t t0 = gtimer();
    while (true) {
      unsigned long long v;
      asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(cnt) : "memory");
      if (v >= target) break;
      if (gtimer() - t0 > kTimeoutNs) {
        record_error(TT_ERR_TIMEOUT, 100);
        *failed = 1;
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
  return *failed == 0;
}

// Compaction position of each middle-rank index (-1 if pruned), from D_d
// (pack) or from the kept list (gather).
__device__ void eng_pos_map(const EngTask& t, int* pos) {
  compaction_map(t.s, t.rd, pos, nullptr, nullptr);
}

// Element f (flat index into dA (N x rd) or dB (rd x M)) read from the
// compacted token sums.
// (32-bit index arithmetic: N*rd and rd*M stay far below 2^31.)
__device__ __forceinline__ float eng_gather(const EngTask& t, const int* pos, int64_t f64) {
  const unsigned f = (unsigned)f64;
  if (t.gather == 1) {
    const unsigned j = f / (unsigned)t.rd;
    const int c = pos[f - j * (unsigned)t.rd];
    return c >= 0 ? __ldcg(t.tc.dAc + (size_t)j * RP + c) : 0.f;
  }
  const unsigned a = f / (unsigned)t.M;
  const int c = pos[a];
  return c >= 0 ? __ldcg(t.tc.dBc + (size_t)(f - a * (unsigned)t.M) * RP + c) : 0.f;
}

// One kET x kET output tile of C over one K slice.
__device__ void eng_gemm_unit(const EngTask& t, int u, float (*As)[kET + 1],
                              float (*Bs)[kET + 1], int* pos, float* ksc, float* csc, int nu) {
  (void)nu;
  if (t.pack_side || t.gather) eng_pos_map(t, pos);
  const GemmArgs& g = t.g;
  const int S = t.splits;
  const int tiles_n = (int)((g.n + kET - 1) / kET);
  const int ks = u % S;
  const int tile = u / S;
  const int64_t m0 = (int64_t)(tile / tiles_n) * kET, n0 = (int64_t)(tile % tiles_n) * kET;
  int64_t chunk = (g.k + S - 1) / S;
  chunk = (chunk + kEK - 1) / kEK * kEK;
  const int64_t kb = (int64_t)ks * chunk;
  const int64_t ke = kb + chunk < g.k ? kb + chunk : g.k;
  const float* A = static_cast<const float*>(g.A);
  const float* B = static_cast<const float*>(g.B);
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  float acc[2][2] = {};
  // the periodic scales of this tile's columns, once per unit
  if (tid < kET) {
    const int64_t gn = n0 + tid;
    csc[tid] = (g.cscale && gn < g.n) ? g.cscale[(unsigned)gn % (unsigned)g.clen] : 1.f;
  }
  for (int64_t k0 = kb; k0 < ke; k0 += kEK) {
    // the K slice's periodic scales, loaded together with the operands
    float kscv = 1.f;
    if (tid < kEK) {
      const int64_t gk = k0 + tid;
      if (g.kscale && gk < ke) kscv = __ldcg(g.kscale + (unsigned)gk % (unsigned)g.klen);
    }
    if (k0 == kb) TLU_STAMP(nu, 3);
    // coalesced loads: walk the operand's unit-stride index fastest (the
    // [kEK][kET+1] tiles are conflict-free either way).  All 2 x 16 loads of
    // a thread are issued before any is used, so they overlap in flight.
    constexpr int kPer = (kET * kEK) / kEngThreads;
    const bool a_kfast = g.sak == 1 && g.sam != 1;
    const bool b_kfast = g.sbk == 1 && g.sbn != 1;
    float va[kPer], vb[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int idx = tid + e * kEngThreads;
      const int a_m = a_kfast ? idx / kEK : idx % kET;
      const int a_k = a_kfast ? idx % kEK : idx / kET;
      const int64_t gm = m0 + a_m, gk = k0 + a_k;
      va[e] = 0.f;
      if (gm < g.m && gk < ke) {
        const int64_t f = gm * g.sam + gk * g.sak;
        va[e] = (t.gather && t.gather_op == 0) ? eng_gather(t, pos, f) : __ldcg(A + f);
      }
      const int b_n = b_kfast ? idx / kEK : idx % kET;
      const int b_k = b_kfast ? idx % kEK : idx / kET;
      const int64_t gn = n0 + b_n, gk2 = k0 + b_k;
      vb[e] = 0.f;
      if (gn < g.n && gk2 < ke) {
        const int64_t f = gk2 * g.sbk + gn * g.sbn;
        vb[e] = (t.gather && t.gather_op == 1) ? eng_gather(t, pos, f) : __ldcg(B + f);
      }
    }
    if (tid < kEK) ksc[tid] = kscv;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int idx = tid + e * kEngThreads;
      const int a_m = a_kfast ? idx / kEK : idx % kET;
      const int a_k = a_kfast ? idx % kEK : idx / kET;
      As[a_k][a_m] = va[e];
      const int b_n = b_kfast ? idx / kEK : idx % kET;
      const int b_k = b_kfast ? idx % kEK : idx / kET;
      Bs[b_k][b_n] = vb[e];
    }
    __syncthreads();
    if (k0 == kb) TLU_STAMP(nu, 4);
    const int kn = (int)(ke - k0 < kEK ? ke - k0 : kEK);
#pragma unroll 8
    for (int kk = 0; kk < kn; ++kk) {
      const float sk = ksc[kk];
      const float a0 = As[kk][ty * 2] * sk, a1 = As[kk][ty * 2 + 1] * sk;
      const float b0 = Bs[kk][tx * 2], b1 = Bs[kk][tx * 2 + 1];
      acc[0][0] = fmaf(a0, b0, acc[0][0]);
      acc[0][1] = fmaf(a0, b1, acc[0][1]);
      acc[1][0] = fmaf(a1, b0, acc[1][0]);
      acc[1][1] = fmaf(a1, b1, acc[1][1]);
    }
    __syncthreads();
    if (k0 == kb) TLU_STAMP(nu, 5);
  }
  float* C = static_cast<float*>(g.C);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int64_t gm = m0 + ty * 2 + i;
    if (gm >= g.m) continue;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int64_t gn = n0 + tx * 2 + j;
      if (gn >= g.n) continue;
      if (S > 1) {
        t.partial[((int64_t)ks * g.m + gm) * g.n + gn] = acc[i][j];
        continue;
      }
      float v = acc[i][j] * csc[tx * 2 + j];
      if (g.rscale) v *= g.rscale[gm];
      const int64_t ci = gm * g.scm + gn * g.scn;
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
            static_cast<__nv_bfloat16*>(t.tc.At)[(size_t)c * t.N + jj] = b;
          }
        } else {
          const unsigned a = cu / (unsigned)t.M;
          const int c = pos[a];
          if (c >= 0) {
            const unsigned o = cu - a * (unsigned)t.M;
            static_cast<__nv_bfloat16*>(t.tc.Bt)[(size_t)o * RP + c] = b;
            static_cast<__nv_bfloat16*>(t.tc.Bm)[(size_t)c * t.M + o] = b;
          }
        }
      }
    }
  }
}

// kEChain unit: prefixes [p0, p0 + pb) of one side's chain and last-mode
// indices [q0, q0 + sb).  One cooperative pass loads everything the unit
// needs into shared memory (the C_0 rows of its prefixes, the inner cores
// C_1..C_{L-2} whole, the C_{L-1}[:, q0:q0+sb, :] slice and the diagonals),
// so the loads are all in flight together; the chain vectors are then
// rebuilt from shared memory.  P_k rows are written once (by the units with
// q0 == 0), the final rows go to `out` and, on the tensor-core path, to the
// compacted bf16 operands.
constexpr int kChainPB = 32;        // max prefixes per unit
constexpr int kChainSmem = 40960;   // floats of dynamic shared memory per CTA

__host__ __device__ inline int64_t chain_stage_floats(const ChainDesc& c) {
  int64_t f = 2 * kChainPB * 64 + kChainPB * (TT_MAX_D + 1) + (int64_t)(c.L > 1 ? c.L - 1 : 0) * 64;
  for (int k = 1; k <= c.L - 2; ++k) f += (int64_t)c.r[k] * c.s[k] * c.r[k + 1];
  f += (int64_t)c.r[c.L - 1] * c.sb * c.r[c.L];
  return f;
}

// Asynchronous 4-byte global -> shared copies: a thread issues all of its
// copies without waiting, so a whole staging pass costs one round trip.
// (Only read-only inputs of the launch are staged this way.)
__device__ __forceinline__ void cp_async4(float* smem, const float* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(su32(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ void eng_chain_unit(const EngTask& t, int u, int* pos, float* dsm, int nu) {
  (void)nu;
  const ChainDesc& c = t.ch;
  const int L = c.L;
  const int pb = c.pb, sb = c.sb;
  const int64_t p0 = (int64_t)(u / c.nsb) * pb;
  const int q0 = (u % c.nsb) * sb;
  const int np = (int)(c.nprefix - p0 < pb ? c.nprefix - p0 : pb);
  const int sl = c.s[L - 1], rl1 = c.r[L - 1], rL = c.r[L];
  const int nq = (sl - q0 < sb ? sl - q0 : sb);
  // shared-memory layout
  float* va = dsm;
  float* vb = va + kChainPB * 64;
  int* dig = reinterpret_cast<int*>(vb + kChainPB * 64);  // [pb][TT_MAX_D + 1] digits, alpha
  float* dg = vb + kChainPB * 64 + kChainPB * (TT_MAX_D + 1);  // [L-1][64] diagonals
  float* cs[TT_MAX_D] = {};                  // staged inner cores
  float* cur = dg + (L > 1 ? L - 1 : 0) * 64;
  for (int k = 1; k <= L - 2; ++k) {
    cs[k] = cur;
    cur += c.r[k] * c.s[k] * c.r[k + 1];
  }
  float* cf = cur;                           // [rl1][nq][rL] final slice
  // prefix digits, 32-bit (prefix counts stay far below 2^31)
  for (int pi = threadIdx.x; pi < np; pi += blockDim.x) {
    unsigned rem = (unsigned)(p0 + pi);
    for (int k = L - 2; k >= 0; --k) {
      dig[pi * (TT_MAX_D + 1) + k] = (int)(rem % (unsigned)c.s[k]);
      rem /= (unsigned)c.s[k];
    }
    dig[pi * (TT_MAX_D + 1) + TT_MAX_D] = (int)rem;  // alpha
  }
  __syncthreads();
  // one asynchronous staging pass for everything the unit reads
  const int r1 = c.r[1];
  for (int e = threadIdx.x; e < np * r1; e += blockDim.x) {
    const int pi = e / r1, col = e - (e / r1) * r1;
    const int alpha = dig[pi * (TT_MAX_D + 1) + TT_MAX_D], d0 = dig[pi * (TT_MAX_D + 1)];
    cp_async4(va + pi * 64 + col, c.core[0] + ((int64_t)(alpha * c.s[0] + d0) * r1 + col));
  }
  for (int k = 0; k < L - 1; ++k)
    for (int e = threadIdx.x; e < c.r[k + 1]; e += blockDim.x) cp_async4(dg + k * 64 + e, c.diag[k] + e);
  for (int k = 1; k <= L - 2; ++k) {
    const int n = c.r[k] * c.s[k] * c.r[k + 1];
    for (int e = threadIdx.x; e < n; e += blockDim.x) cp_async4(cs[k] + e, c.core[k] + e);
  }
  {
    const int n = rl1 * nq * rL;
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
      const int col = e % rL;
      const int qi = (e / rL) % nq;
      const int b = e / (rL * nq);
      cp_async4(cf + e, c.core[L - 1] + ((int64_t)b * sl + q0 + qi) * rL + col);
    }
  }
  if (t.pack_side) compaction_map(t.s, t.rd, pos, nullptr, nullptr);
  cp_async_wait_all();
  __syncthreads();
  TLU_STAMP(nu, 3);
  TLU_STAMP(nu, 4);
  // steps 1 .. L-2: v <- (v * E_{k-1}) . C_k[:, s_k, :]
  for (int k = 1; k <= L - 2; ++k) {
    const int rk = c.r[k], rk1 = c.r[k + 1], sk = c.s[k];
    const float* Ek = dg + (k - 1) * 64;
    for (int e = threadIdx.x; e < np * rk1; e += blockDim.x) {
      const int pi = e / rk1, col = e - (e / rk1) * rk1;
      const int* dd = dig + pi * (TT_MAX_D + 1);
      int64_t row = dd[TT_MAX_D];
      for (int kk = 0; kk <= k; ++kk) row = row * c.s[kk] + dd[kk];
      const float* Ck = cs[k] + dd[k] * rk1 + col;
      const float* v = va + pi * 64;
      float a0 = 0.f, a1 = 0.f;
      int b = 0;
      for (; b + 1 < rk; b += 2) {
        a0 = fmaf(v[b] * Ek[b], Ck[b * sk * rk1], a0);
        a1 = fmaf(v[b + 1] * Ek[b + 1], Ck[(b + 1) * sk * rk1], a1);
      }
      if (b < rk) a0 = fmaf(v[b] * Ek[b], Ck[b * sk * rk1], a0);
      const float acc = a0 + a1;
      vb[pi * 64 + col] = acc;
      if (q0 == 0 && c.prow[k]) c.prow[k][row * rk1 + col] = acc;
    }
    __syncthreads();
    float* tmp = va;
    va = vb;
    vb = tmp;
  }
  TLU_STAMP(nu, 5);
  // final rows (prefix, q) = (v * E_{L-2}) . C_{L-1}[:, q, :]
  const float* EL = dg + (L - 2) * 64;
  const int nout = np * nq * rL;
  for (int e = threadIdx.x; e < nout; e += blockDim.x) {
    const int col = e % rL;
    const int qi = (e / rL) % nq;
    const int pi = e / (rL * nq);
    const float* v = va + pi * 64;
    const float* Cq = cf + qi * rL + col;
    float a0 = 0.f, a1 = 0.f;
    int b = 0;
    for (; b + 1 < rl1; b += 2) {
      a0 = fmaf(v[b] * EL[b], Cq[b * nq * rL], a0);
      a1 = fmaf(v[b + 1] * EL[b + 1], Cq[(b + 1) * nq * rL], a1);
    }
    if (b < rl1) a0 = fmaf(v[b] * EL[b], Cq[b * nq * rL], a0);
    const float acc = a0 + a1;
    const int64_t f = ((p0 + pi) * sl + q0 + qi) * rL + col;  // flat index into P_{L-1}
    c.out[f] = acc;
    if (t.pack_side) {
      const __nv_bfloat16 bv = __float2bfloat16_rn(acc);
      if (t.pack_side == 1) {  // A (N x rd): f = j * rd + a
        const unsigned jj = (unsigned)f / (unsigned)t.rd;
        const int cc = pos[(unsigned)f - jj * (unsigned)t.rd];
        if (cc >= 0) {
          static_cast<__nv_bfloat16*>(t.tc.Anr)[(size_t)jj * RP + cc] = bv;
          static_cast<__nv_bfloat16*>(t.tc.At)[(size_t)cc * t.N + jj] = bv;
        }
      } else {  // B (rd x M): f = a * M + o
        const unsigned a = (unsigned)f / (unsigned)t.M;
        const int cc = pos[a];
        if (cc >= 0) {
          const unsigned o = (unsigned)f - a * (unsigned)t.M;
          static_cast<__nv_bfloat16*>(t.tc.Bt)[(size_t)o * RP + cc] = bv;
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
  float v = 0.f;
  for (int ks = 0; ks < t.splits; ++ks) v += __ldcg(t.partial + (int64_t)ks * g.m * g.n + i);
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
  const int64_t base = (int64_t)u * 1024;
  for (int e = threadIdx.x; e < 1024; e += blockDim.x) {
    const int64_t i = base + e;
    if (i >= t.n) break;
    float v = t.x ? __ldcg(t.x + i) : 0.f;
    if (t.s) v *= t.s[(unsigned)i % (unsigned)t.len];
    t.out[i] = t.acc ? __ldcg(t.out + i) + v : v;
  }
}

__global__ void __launch_bounds__(kEngThreads) eng_kernel(const __grid_constant__ EngProgram prog) {
  extern __shared__ float eng_dsm[];  // kChainSmem floats, used by kEChain units
  __shared__ float As[kEK][kET + 1];
  __shared__ float Bs[kEK][kET + 1];
  __shared__ float red[32];
  __shared__ int pos[RP];
  __shared__ float ksc[kEK];
  __shared__ float csc[kET];
  __shared__ __align__(16) EngProgram p;  // the whole program, copied once per CTA
  __shared__ int failed;
  pdl_wait();  // params and workspace may be written by the previous grid
  pdl_trigger();
  {
    const uint4* src = reinterpret_cast<const uint4*>(&prog);
    uint4* dst = reinterpret_cast<uint4*>(&p);
    for (int i = threadIdx.x; i < (int)(sizeof(EngProgram) / 16); i += blockDim.x) dst[i] = src[i];
  }
  if (threadIdx.x == 0) {
    failed = 0;
    TL_STAMP(2, 0);
  }
  __syncthreads();
#ifdef TTC_TIMELINE
  int nu = 0;
#endif
  for (int ph = 0; ph < p.nphases; ++ph) {
    const int t0 = p.phase_begin[ph], t1 = p.phase_begin[ph + 1];
    int total = 0;
    for (int t = t0; t < t1; ++t) total += p.t[t].units;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
      int t = t0, uu = u;
      while (uu >= p.t[t].units) uu -= p.t[t++].units;
      const EngTask& k = p.t[t];
#ifdef TTC_TIMELINE
      if (threadIdx.x == 0 && nu < 8) {
        g_tlu[blockIdx.x & 255][nu][0] = ph * 100 + t;
        g_tlu[blockIdx.x & 255][nu][1] = gtimer();
      }
#endif
      switch (k.kind) {
        case kEGemm:
#ifdef TTC_TIMELINE
          eng_gemm_unit(k, uu, As, Bs, pos, ksc, csc, nu);
#else
          eng_gemm_unit(k, uu, As, Bs, pos, ksc, csc, 0);
#endif
          break;
        case kEGemmFinal: eng_gemm_final_unit(k, uu); break;
        case kEColdot: eng_coldot_unit(k, uu, red); break;
        case kEScale: eng_scale_unit(k, uu); break;
        case kEPack:
          tc_pack_unit(k.A, k.B, k.s, k.rd, k.N, k.M, k.tc, k.zero, k.pad_only, uu);
          break;
        case kEDd:
          tc_dd_unit(k.tc, k.s, k.rd, k.out, k.acc);
          break;
        case kEChain:
#ifdef TTC_TIMELINE
          eng_chain_unit(k, uu, pos, eng_dsm, nu);
#else
          eng_chain_unit(k, uu, pos, eng_dsm, 0);
#endif
          break;
        case kEUnpack:
          tc_unpack_unit(k.tc, k.s, k.rd, k.N, k.M, k.dA, k.dB, k.out, k.acc, uu);
          break;
        default: break;
      }
#ifdef TTC_TIMELINE
      __syncthreads();
      if (threadIdx.x == 0 && nu < 8) g_tlu[blockIdx.x & 255][nu][2] = gtimer();
      ++nu;
#endif
    }
    if (threadIdx.x == 0) TL_STAMP(2, 1 + 2 * ph);
    if (ph + 1 < p.nphases && !eng_grid_barrier(p.slot, gridDim.x, &failed)) return;
    if (threadIdx.x == 0) TL_STAMP(2, 2 + 2 * ph);
  }
}

}  // namespace

// ---- host side -------------------------------------------------------------

void EngBuilder::begin_phase() {
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

void EngBuilder::end() { p.phase_begin[p.nphases] = p.ntasks; }

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t eng_partial_floats(int64_t m, int64_t n, int64_t k) {
  (void)k;
  return (size_t)(m * n) * 16;  // at most 16 K-splits
}

void eng_gemm_task(EngTask* t, const GemmArgs& g, float* partial_ws, size_t partial_cap) {
  t->kind = kEGemm;
  t->g = g;
  const int64_t tiles = ceil_div(g.m, kET) * ceil_div(g.n, kET);
  int64_t splits = 1;
  // split long reductions so that a phase has a few units per SM and each
  // unit still walks at least a few K slices
  if (partial_ws && tiles < 256) {
    const int64_t want = ceil_div(256, tiles);
    const int64_t maxs = ceil_div(g.k, kEK);
    splits = want < maxs ? want : maxs;
    if (splits > 16) splits = 16;
    if ((size_t)(splits * g.m * g.n) > partial_cap) splits = 1;
    if (splits < 1) splits = 1;
  }
  t->splits = (int)splits;
  t->partial = splits > 1 ? partial_ws : nullptr;
  t->units = (int)(tiles * splits);
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
  t->units = (int)ceil_div((L.N + L.M) * RP + RP, kPackPer);
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
  t->units = (int)ceil_div((L.N + L.M) * L.rd + L.rd, kPackPer);
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

cudaError_t eng_launch(const EngProgram& prog, cudaStream_t st) {
  static std::atomic<unsigned> next_slot{0};
  static int grid = 0;
  if (!grid) {
    int dev = 0, sms = 0, per = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaFuncSetAttribute(eng_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kChainSmem * sizeof(float))) != cudaSuccess)
      return cudaErrorLaunchFailure;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, eng_kernel, kEngThreads,
                                                  kChainSmem * sizeof(float));
    grid = sms * (per > 0 ? 1 : 0);
    if (grid <= 0) return cudaErrorLaunchFailure;
  }
  EngProgram p = prog;
  p.slot = next_slot.fetch_add(1) % kBarSlots;
  int g = grid;
  bool coop = true;
#ifdef TTC_TIMELINE
  // measurement builds only: grid size and launch kind from the environment
  if (const char* e = getenv("TTC_ENG_GRID")) g = atoi(e) > 0 && atoi(e) < grid ? atoi(e) : grid;
  if (getenv("TTC_ENG_NONCOOP")) coop = false;
#endif
  cudaError_t e = launch_ex(eng_kernel, dim3(g), dim3(kEngThreads), kChainSmem * sizeof(float), st,
                            coop, p);
  count_launches(1);
  return e;
}

}  // namespace ttc
