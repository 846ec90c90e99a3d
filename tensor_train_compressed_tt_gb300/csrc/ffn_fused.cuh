// Fused FFN pair on the tensor cores: y = TT_down(GELU(TT_up(x))) for bf16
// activations, with the hidden activations h = TT_up(x) and a = GELU(h) (and,
// in the backward, da and dh) kept on the SM: TMEM accumulators and bf16
// tiles in shared memory, one 128-column hidden chunk at a time.  Included
// once, by tc_fused.cu, after the single-layer kernels (it uses their PTX
// helpers and the per-device status word).
//
// Per tile of 128 tokens (the layer shapes of the CoMERA project page's
// feed-forward rows, "Results", rank table: 768 -> 3072 -> 768 at rank 30):
//   z1 = x A1                 (x streamed, 128 features a chunk)
//   z1' = z1 diag(D1)         -> bf16 tile
//   for each 128-column chunk c of the hidden width:
//     h_c  = z1' B1[:, c]     (TMEM, double-buffered)
//     a_c  = GELU(h_c)        -> bf16 tile (epilogue warps)
//     z2  += a_c A2[c, :]     (TMEM)
//   z2' = z2 diag(D2)         -> bf16 tile
//   y   = z2' B2              (128 outputs a chunk, TMA stores)
// GELU is the erf form h Phi(h) with erf(u / sqrt 2) evaluated as
// tanh(sqrt(2/pi) (u + 0.044715 u^3)) (the tanh approximation of Hendrycks
// and Gimpel's GELU paper: |Phi error| <= 1.8e-4, |GELU error| <= 4.8e-4,
// far below a bf16 rounding), tanh by the hardware's tanh.approx.f32.
#pragma once

namespace ttc {
namespace {

constexpr int FFN_NST_F = 3;  // forward ring stages
constexpr int FFN_NST_B = 2;  // backward ring stages (shared memory holds four tiles more)

__device__ __forceinline__ float tanh_hw(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kGeluK = 0.79788456080286536f;                 // sqrt(2 / pi)
constexpr float kGeluKC = 0.79788456080286536f * 0.044715f;    // sqrt(2 / pi) * 0.044715

// GELU(u) = u Phi(u), Phi(u) ~ (1 + tanh(k (u + c u^3))) / 2, and with it
// g = da * GELU'(u) of the same approximation,
// GELU'(u) = (1 + t) / 2 + (u / 2)(1 - t^2) k (1 + 3 c u^2), t = tanh(k (u + c u^3)).
// Both for a pair of elements in packed f32x2 arithmetic (two FMAs an
// instruction on this architecture, each rounded as a scalar FMA); the tanh
// stays one special-function operation an element.
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 gelu_tanh2(float2 u) {
  const float2 arg = __fmul2_rn(u, __ffma2_rn(f2(kGeluKC), __fmul2_rn(u, u), f2(kGeluK)));
  const float2 t = make_float2(tanh_hw(arg.x), tanh_hw(arg.y));
  const float2 hu = __fmul2_rn(f2(0.5f), u);
  return __ffma2_rn(hu, t, hu);
}
__device__ __forceinline__ void gelu_tanh_grad2(float2 u, float2 da, float2& a, float2& g) {
  const float2 u2 = __fmul2_rn(u, u);
  const float2 arg = __fmul2_rn(u, __ffma2_rn(f2(kGeluKC), u2, f2(kGeluK)));
  const float2 t = make_float2(tanh_hw(arg.x), tanh_hw(arg.y));
  const float2 hu = __fmul2_rn(f2(0.5f), u);
  a = __ffma2_rn(hu, t, hu);
  const float2 dq = __ffma2_rn(f2(3.f * kGeluKC), u2, f2(kGeluK));
  const float2 omt = __ffma2_rn(make_float2(-t.x, -t.y), t, f2(1.f));
  const float2 d = __ffma2_rn(__fmul2_rn(hu, omt), dq, __ffma2_rn(f2(0.5f), t, f2(0.5f)));
  g = __fmul2_rn(da, d);
}

// Throughput probe of the fused FFN kernels' GELU arithmetic (a measurement
// hook): every thread carries eight pairs of values through `iters` rounds of
// GELU (mode 0, the forward's) or GELU and GELU' (mode 1, the backward's),
// each result feeding the next round, entirely in registers, and writes one
// sum so that nothing is dropped.  16 evaluations a thread a round.
__global__ void __launch_bounds__(256) gelu_rate_kernel(int mode, int iters, float* out) {
  float2 v[8], w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float base = (float)((threadIdx.x * 8 + j) % 61) * 0.1f - 3.f;  // in [-3, 3]
    v[j] = make_float2(base, base + 0.05f);
    w[j] = make_float2(1.f, 0.5f);
  }
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (mode == 0) {
        const float2 a = gelu_tanh2(v[j]);
        v[j] = __ffma2_rn(a, f2(0.9f), f2(-0.2f));  // stays in about [-3, 3]
      } else {
        float2 a, g;
        gelu_tanh_grad2(v[j], w[j], a, g);
        v[j] = __ffma2_rn(a, f2(0.9f), f2(-0.2f));
        w[j] = __ffma2_rn(g, f2(0.5f), f2(0.5f));
      }
    }
  }
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) sum += v[j].x + v[j].y + w[j].x + w[j].y;
  out[blockIdx.x * blockDim.x + threadIdx.x] = sum;
}

// Per-warp stamps of CTA 0 (timeline builds only): [kernel][warp][slot]
#ifdef TTC_TIMELINE
__device__ unsigned long long g_tlw[2][16][48];
#define TLW(k, slot) \
  if (blockIdx.x == 0 && (threadIdx.x & 31) == 0 && (slot) < 48) g_tlw[(k)][threadIdx.x >> 5][(slot)] = gtimer()
#else
#define TLW(k, slot) ((void)0)
#endif

struct FfnFwdArgs {
  int64_t T;
  int nN, nH, nM, ntiles;
  int kb1, kb2;     // 16-wide K blocks that cover the middle ranks (the rest is zero padding)
  int nr;           // MMA width of the rank dimension: 32 when both middle ranks are <= 32, else 64
  int save_z;       // keep z1' and z2' (bf16 [T][64] each) for the backward
  int M;
  int prefetch_x;   // x of the first stages requested before the dependency wait
  const float* Dc1;
  const float* Dc2;
};

struct FfnFwdSmem {
  uint64_t full[FFN_NST_F], empty[FFN_NST_F];
  uint64_t z1_full, z1_empty, z2_full, z2_empty, zp_full, zp_empty;
  uint64_t h_full[2], h_empty[2], a_full, a_empty, stg_free, fin;
  uint32_t tmem_base;
  int abort_flag;
  float Dc1[RP], Dc2[RP];
};

// TMEM columns of the forward
constexpr uint32_t FF_Z1 = 0, FF_Z2 = 64, FF_H = 128;  // H: two 128-column buffers

constexpr size_t kSmemFfnFwd =
    FFN_NST_F * STAGE + BOX + 2 * BOX + sizeof(FfnFwdSmem) + 1024;
static_assert(kSmemFfnFwd <= 227 * 1024, "FFN forward smem");

// Ring items in the producer's order, per tile: nN x items (two x boxes +
// the A1 rows of the chunk), nH hidden items (the A2 rows of the chunk at
// +0, the B1 columns at +OPND), nM output items (the B2 columns at +OPND).
__global__ void __launch_bounds__(NTHREADS, 1)
    ffn_fwd_kernel(const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_anr1,
                   const __grid_constant__ CUtensorMap tm_bm1,
                   const __grid_constant__ CUtensorMap tm_anr2,
                   const __grid_constant__ CUtensorMap tm_bm2,
                   const __grid_constant__ CUtensorMap tm_y,
                   const __grid_constant__ CUtensorMap tm_zs1,
                   const __grid_constant__ CUtensorMap tm_zs2, FfnFwdArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1k(smem_raw);
  uint8_t* stages = base;
  uint8_t* zp = base + FFN_NST_F * STAGE;  // z1' tile, then z2' tile
  uint8_t* atile = zp + BOX;               // a_c: [128 tokens][128 hidden] as two boxes;
                                           // the y staging boxes after the hidden loop
  FfnFwdSmem& S = *reinterpret_cast<FfnFwdSmem*>(atile + 2 * BOX);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < FFN_NST_F; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.z1_full, 1);
    mbar_init(&S.z1_empty, NEPI);
    mbar_init(&S.z2_full, 1);
    mbar_init(&S.z2_empty, NEPI);
    mbar_init(&S.zp_full, NEPI);
    mbar_init(&S.zp_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.h_full[b], 1);
      mbar_init(&S.h_empty[b], NEPI);
    }
    mbar_init(&S.a_full, NEPI);
    mbar_init(&S.a_empty, 1);
    mbar_init(&S.stg_free, NEPI);
    mbar_init(&S.fin, 1);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int s = 0; s < fwd_prefetched(p, FFN_NST_F); ++s) {  // x of the first chunks
      uint8_t* st = stages + s * STAGE;
      mbar_expect_tx(&S.full[s], 3 * BOX);
      tma_load(st, &tm_x, &S.full[s], s * CH, blockIdx.x * TILE);
      tma_load(st + BOX, &tm_x, &S.full[s], s * CH + 64, blockIdx.x * TILE);
    }
  }
  if (warp == 1) tmem_alloc(&S.tmem_base);
  pdl_wait();  // nothing a previous grid writes is touched before this point (but x above)
  pdl_trigger();
  if (threadIdx.x < RP) {
    S.Dc1[threadIdx.x] = p.Dc1[threadIdx.x];
    S.Dc2[threadIdx.x] = p.Dc2[threadIdx.x];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;
  const int nitems = p.nN + p.nH + p.nM;
  if (threadIdx.x == 0) TL_STAMP(0, 0);

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int it = 0;
      int last_parity[FFN_NST_F];
      for (int s = 0; s < FFN_NST_F; ++s) last_parity[s] = -1;
      bool ok = true;
      const int npre = fwd_prefetched(p, FFN_NST_F);  // x already requested
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x) {
        const int tok0 = tile * TILE;
        for (int c = 0; c < nitems; ++c, ++it) {
          const int s = it % FFN_NST_F;
          const uint32_t ph = (it / FFN_NST_F) & 1;
          if (!wait_bar(&S.empty[s], ph ^ 1, abort_flag, 50)) { ok = false; break; }
          uint8_t* st = stages + s * STAGE;
          if (it < npre) {
            tma_load(st + OPND, &tm_anr1, &S.full[s], 0, c * CH);
          } else if (c < p.nN) {
            mbar_expect_tx(&S.full[s], 3 * BOX);
            tma_load(st, &tm_x, &S.full[s], c * CH, tok0);
            tma_load(st + BOX, &tm_x, &S.full[s], c * CH + 64, tok0);
            tma_load(st + OPND, &tm_anr1, &S.full[s], 0, c * CH);
          } else if (c < p.nN + p.nH) {
            // chunk order rotated by the tile index: concurrent CTAs read
            // different operand chunks instead of all the same lines of L2
            const int hc = rot_chunk(c - p.nN, p.nH, tile);
            mbar_expect_tx(&S.full[s], 2 * BOX);
            tma_load(st, &tm_anr2, &S.full[s], 0, hc * CH);  // [128 hidden][64 ranks]
            tma_load(st + OPND, &tm_bm1, &S.full[s], hc * CH, 0);
            tma_load(st + OPND + BOX / 2, &tm_bm1, &S.full[s], hc * CH + 64, 0);
          } else {
            const int oc = c - p.nN - p.nH;
            mbar_expect_tx(&S.full[s], BOX);
            tma_load(st + OPND, &tm_bm2, &S.full[s], oc * CH, 0);
            tma_load(st + OPND + BOX / 2, &tm_bm2, &S.full[s], oc * CH + 64, 0);
          }
          last_parity[s] = (int)ph;
        }
      }
      for (int s = 0; s < FFN_NST_F; ++s)
        if (last_parity[s] >= 0) drain_bar(&S.full[s], (uint32_t)last_parity[s]);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_z = idesc(128, p.nr, 0, 1);  // B = rows [K][64 ranks], MN-major
      const uint32_t id_h = idesc(128, 128, 0, 1);  // B = [64 ranks][128 columns], MN-major
      const uint32_t zp_addr = su32(zp);
      const uint32_t at_addr = su32(atile);
      int it = 0, hc = 0, ac = 0, tl = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x, ++tl) {
        // z1 = x A1
        if (!wait_bar(&S.z1_empty, (tl & 1) ^ 1, abort_flag, 51)) break;
        tc_fence_after();
        for (int c = 0; c < p.nN; ++c, ++it) {
          const int s = it % FFN_NST_F;
          if (!wait_bar(&S.full[s], (it / FFN_NST_F) & 1, abort_flag, 52)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma(tmem + FF_Z1, kdesc(st + b * BOX) + 2 * k,
                  mndesc(st + OPND + b * (BOX / 2), 1024) + 128 * k, id_z, (c | b | k) != 0);
          mma_commit(&S.empty[s]);
        }
        if (!ok) break;
        mma_commit(&S.z1_full);
        // hidden chunks: h_c = z1' B1[:, c]; z2 += a_c A2[c, :] one chunk behind
        if (!wait_bar(&S.zp_full, 0, abort_flag, 53)) break;  // z1' tile written
        tc_fence_after();
        if (p.save_z) {
          tma_store(&tm_zs1, zp, 0, tile * TILE);
          bulk_commit();
        }
        if (!wait_bar(&S.z2_empty, (tl & 1) ^ 1, abort_flag, 54)) break;
        const int ih = it;
        // h_c = z1' B1[:, c] into H buffer c & 1, issued two chunks ahead of
        // the z2 product that consumes GELU(h_c), so the epilogue finds the
        // next h ready when it finishes a chunk
        auto issue_h = [&](int c) -> bool {
          const int s = (ih + c) % FFN_NST_F;
          const int hb = hc & 1;
          if (!wait_bar(&S.full[s], ((ih + c) / FFN_NST_F) & 1, abort_flag, 55)) return false;
          if (!wait_bar(&S.h_empty[hb], ((hc >> 1) & 1) ^ 1, abort_flag, 56)) return false;
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
          for (int k = 0; k < p.kb1; ++k)
            mma(tmem + FF_H + hb * 128, kdesc(zp_addr) + 2 * k,
                mndesc(st + OPND, BOX / 2) + 128 * k, id_h, k != 0);
          mma_commit(&S.h_full[hb]);
          if (tl == 0 && c < 8) TLW(0, 2 * c);
          ++hc;
          if (c == p.nH - 1) {  // the z1' tile's last reader is issued
            if (p.save_z) bulk_wait_read<0>();
            mma_commit(&S.zp_empty);
          }
          return true;
        };
        if (!issue_h(0) || (p.nH > 1 && !issue_h(1))) break;
        for (int c = 0; c < p.nH; ++c) {
          const int s = (ih + c) % FFN_NST_F;
          if (!wait_bar(&S.a_full, ac & 1, abort_flag, 57)) { ok = false; break; }
          if (tl == 0 && c < 8) TLW(0, 2 * c + 1);
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma(tmem + FF_Z2, kdesc(at_addr + b * BOX) + 2 * k,
                  mndesc(st + b * (BOX / 2), 1024) + 128 * k, id_z, (c | b | k) != 0);
          mma_commit(&S.a_empty);
          mma_commit(&S.empty[s]);
          ++ac;
          if (c + 2 < p.nH && !issue_h(c + 2)) { ok = false; break; }
        }
        if (!ok) break;
        it = ih + p.nH;
        mma_commit(&S.z2_full);
        // y = z2' B2
        if (!wait_bar(&S.zp_full, 1, abort_flag, 58)) break;  // z2' tile written
        tc_fence_after();
        if (p.save_z) {
          tma_store(&tm_zs2, zp, 0, tile * TILE);
          bulk_commit();
        }
        for (int c = 0; c < p.nM; ++c, ++it) {
          const int s = it % FFN_NST_F;
          const int hb = hc & 1;
          if (!wait_bar(&S.h_empty[hb], ((hc >> 1) & 1) ^ 1, abort_flag, 59)) { ok = false; break; }
          if (!wait_bar(&S.full[s], (it / FFN_NST_F) & 1, abort_flag, 60)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
          for (int k = 0; k < p.kb2; ++k)
            mma(tmem + FF_H + hb * 128, kdesc(zp_addr) + 2 * k,
                mndesc(st + OPND, BOX / 2) + 128 * k, id_h, k != 0);
          mma_commit(&S.empty[s]);
          mma_commit(&S.h_full[hb]);
          ++hc;
        }
        if (!ok) break;
        if (p.save_z) bulk_wait_read<0>();
        mma_commit(&S.zp_empty);
      }
      if (p.save_z) bulk_wait_all();
      mma_commit(&S.fin);
      drain_bar(&S.fin, 0);
    }
  } else {
    // ---------------- epilogue: 8 warps, thread = (token row, column half)
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int row = 32 * q + lane;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    uint8_t* my_stg = atile + (warp - 2) * STG;
    int hc = 0, ac = 0, tl = 0;
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++tl) {
      float v[32], w[32];
      bool ok = true;
      // E1: z1' = z1 D1 -> tile
      if (!warp_wait(&S.z1_full, tl & 1, abort_flag, 61)) break;
      if (warp == 2 && lane == 0 && tl == 0) TL_STAMP(0, 1);
      tc_fence_after();
      if (32 * h < p.nr) tmem_ld32(tmem + lane_off + FF_Z1 + 32 * h, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.z1_empty);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 32 * h < p.nr ? v[j] * S.Dc1[32 * h + j] : 0.f;
      if (!warp_wait(&S.zp_empty, 1, abort_flag, 62)) break;
      st_tile_half(zp, row, h, v);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.zp_full);
      // the previous tile's y stores have read their staging boxes (in the A tile)
      if (tl > 0 && !warp_wait(&S.stg_free, (tl - 1) & 1, abort_flag, 63)) break;
      // E2: a_c = GELU(h_c) -> A tile
      for (int c = 0; c < p.nH; ++c) {
        const int hb = hc & 1;
        if (!warp_wait(&S.h_full[hb], (hc >> 1) & 1, abort_flag, 64)) { ok = false; break; }
        if (warp == 2 && lane == 0 && tl == 0 && c < 3) TL_STAMP(0, 2 + 3 * c);
        if (tl == 0 && c < 8) TLW(0, 4 * c);
        tc_fence_after();
        tmem_ld32(tmem + lane_off + FF_H + hb * 128 + 64 * h, v);
        tmem_ld32(tmem + lane_off + FF_H + hb * 128 + 64 * h + 32, w);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.h_empty[hb]);
        ++hc;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float2 gv = gelu_tanh2(make_float2(v[j], v[j + 1]));
          const float2 gw = gelu_tanh2(make_float2(w[j], w[j + 1]));
          v[j] = gv.x;
          v[j + 1] = gv.y;
          w[j] = gw.x;
          w[j + 1] = gw.y;
        }
        if (warp == 2 && lane == 0 && tl == 0 && c < 3) TL_STAMP(0, 3 + 3 * c);
        if (tl == 0 && c < 8) TLW(0, 4 * c + 1);
        if (!warp_wait(&S.a_empty, (ac & 1) ^ 1, abort_flag, 65)) { ok = false; break; }
        if (warp == 2 && lane == 0 && tl == 0 && c < 3) TL_STAMP(0, 4 + 3 * c);
        if (tl == 0 && c < 8) TLW(0, 4 * c + 2);
        st_tile_half(atile + h * BOX, row, 0, v);
        st_tile_half(atile + h * BOX, row, 1, w);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.a_full);
        if (tl == 0 && c < 8) TLW(0, 4 * c + 3);
        ++ac;
      }
      if (!ok) break;
      // E3: z2' = z2 D2 -> tile
      if (!warp_wait(&S.z2_full, tl & 1, abort_flag, 66)) break;
      if (warp == 2 && lane == 0 && tl == 0) TL_STAMP(0, 11);
      tc_fence_after();
      if (32 * h < p.nr) tmem_ld32(tmem + lane_off + FF_Z2 + 32 * h, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.z2_empty);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 32 * h < p.nr ? v[j] * S.Dc2[32 * h + j] : 0.f;
      if (!warp_wait(&S.zp_empty, 0, abort_flag, 67)) break;
      st_tile_half(zp, row, h, v);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.zp_full);
      // E4: y chunks, staged in this warp's box of the A tile (its readers,
      // the z2 MMAs, are done: z2_full came after them)
      for (int c = 0; c < p.nM; ++c) {
        const int hb = hc & 1;
        if (!warp_wait(&S.h_full[hb], (hc >> 1) & 1, abort_flag, 68)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) bulk_wait_read<0>();  // the previous store has read the box
        __syncwarp();
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {
          tmem_ld32(tmem + lane_off + FF_H + hb * 128 + 64 * h + 32 * piece, v);
          stage_bf16_32(my_stg, lane, piece, v);
        }
        tc_fence_before();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&S.h_empty[hb]);
          const int col = c * CH + 64 * h;
          if (col < p.M && (int64_t)tile * TILE + 32 * q < p.T) {
            tma_store(&tm_y, my_stg, col, tile * TILE + 32 * q);
            bulk_commit();
          }
        }
        ++hc;
      }
      if (!ok) break;
      if (warp == 2 && lane == 0 && tl == 0) TL_STAMP(0, 12);
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.stg_free);
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) TL_STAMP(0, 13);
  if (warp == 1) tmem_free(tmem);
}

// Store 32 bf16 values (16 packed words) as columns [32 hh, 32 hh + 32) of
// row `row` of a [128][64] swizzled tile.
__device__ __forceinline__ void st_tile_half_u(uint8_t* tile, int row, int hh,
                                               const uint32_t (&u)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int chunk = (4 * hh + q) ^ (row & 7);
    *reinterpret_cast<uint4*>(tile + row * 128 + chunk * 16) =
        make_uint4(u[4 * q], u[4 * q + 1], u[4 * q + 2], u[4 * q + 3]);
  }
}

struct FfnBwdArgs {
  int64_t T;
  int nN, nH, nM, ntiles;
  int kb1, kb2;
  int nr;  // as in FfnFwdArgs; 32 also splits each W drain to one warp half
  int N, H, M;
  const float* Dc1;
  const float* Dc2;
  const int* rinfo1;  // [0] = compacted middle rank of the up layer
  const int* rinfo2;
  float* dDc1;        // token sums of z1 * dz1' and z2 * dz2'
  float* dDc2;
  ZeroList zero;      // ranges set to 0 on the way (what each layer's merge backward
                      // adds into)
  // TT_DETERMINISTIC: every token sum goes to this CTA's own slot (rows
  // blockIdx.x * rows.. of the four dA / dB maps; dD into dDslot[CTA][quadrant]),
  // stored by the CTA's first tile and added to by its later ones in tile
  // order; the slots are then summed in CTA order
  int det;
  float* dDslot1;
  float* dDslot2;
};

struct FfnBwdSmem {
  uint64_t full[FFN_NST_B], empty[FFN_NST_B];
  uint64_t zl_full, zt_empty, dzp2_full, dzp2_empty, zp2_free, dz2_full;
  uint64_t hd_full, hd_empty, ad_full, ad_empty;
  uint64_t w_full[2], w_empty[2], x_full[2], x_empty[2];
  uint64_t dz1p_full, dz1p_empty, dz1_full, fin;
  uint32_t tmem_base;
  int abort_flag;
  float Dc1[RP], Dc2[RP];
};

// TMEM columns of the backward
constexpr uint32_t FB_H = 0, FB_DA = 128, FB_W = 256, FB_DZ1P = 384, FB_DZ2P = 448;
constexpr uint32_t FB_X = 0;  // phase C: two 128-column dx buffers over H and DA

constexpr size_t kSmemFfnBwd =
    FFN_NST_B * STAGE + 2 * BOX + 4 * BOX + NEPI * STG + sizeof(FfnBwdSmem) + 1024;
static_assert(kSmemFfnBwd <= 227 * 1024, "FFN backward smem");

// Per tile of 128 tokens, with the forward's z1' and z2' tiles loaded:
//   B  dz2' = dy B2^T ; dB2^T += dy^T z2'             (dy streamed)
//      dD2 += sum_t z2 dz2' ; dz2 = dz2' diag(D2)
//   for each 128-column hidden chunk c:
//      h_c = z1' B1[:, c] ; da_c = dz2 A2[c, :]^T       (recomputed, TMEM)
//      a_c = GELU(h_c) ; dh_c = da_c GELU'(h_c)        (epilogue warps -> bf16 tiles)
//      dA2[c] += a_c^T dz2 ; dz1' += dh_c B1[:, c]^T ; dB1^T[c] += dh_c^T z1'
//   dD1 += sum_t z1 dz1' ; dz1 = dz1' diag(D1)
//   C  dx = dz1 A1^T ; dA1 += x^T dz1                  (x streamed)
// The token sums go out by TMA bulk reduce-add (dA / dB) and atomics (dD).
// Ring items per tile: nM dy items (dy boxes + B2 columns), nH hidden items
// (A2 rows at +0, B1 columns at +OPND), nN x items (x boxes + A1 rows).
__global__ void __launch_bounds__(NTHREADS, 1)
    ffn_bwd_kernel(const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_dy,
                   const __grid_constant__ CUtensorMap tm_anr1,
                   const __grid_constant__ CUtensorMap tm_bm1,
                   const __grid_constant__ CUtensorMap tm_anr2,
                   const __grid_constant__ CUtensorMap tm_bm2,
                   const __grid_constant__ CUtensorMap tm_dx,
                   const __grid_constant__ CUtensorMap tm_dac1,
                   const __grid_constant__ CUtensorMap tm_dbc1,
                   const __grid_constant__ CUtensorMap tm_dac2,
                   const __grid_constant__ CUtensorMap tm_dbc2,
                   const __grid_constant__ CUtensorMap tm_zs1,
                   const __grid_constant__ CUtensorMap tm_zs2, FfnBwdArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1k(smem_raw);
  uint8_t* stages = base;
  uint8_t* zt1 = base + FFN_NST_B * STAGE;  // z1', then dz1
  uint8_t* zt2 = zt1 + BOX;                 // z2', then dz2
  uint8_t* atile = zt2 + BOX;               // a_c  [128 tokens][128 hidden], two boxes
  uint8_t* dhtile = atile + 2 * BOX;        // dh_c [128 tokens][128 hidden], two boxes
  uint8_t* staging = dhtile + 2 * BOX;      // one box per epilogue warp
  FfnBwdSmem& S = *reinterpret_cast<FfnBwdSmem*>(staging + NEPI * STG);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < FFN_NST_B; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.zl_full, 1);
    mbar_init(&S.zt_empty, 1);
    mbar_init(&S.dzp2_full, 1);
    mbar_init(&S.dzp2_empty, NEPI);
    mbar_init(&S.zp2_free, 1);
    mbar_init(&S.dz2_full, NEPI);
    mbar_init(&S.hd_full, 1);
    mbar_init(&S.hd_empty, NEPI);
    mbar_init(&S.ad_full, NEPI);
    mbar_init(&S.ad_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.w_full[b], 1);
      mbar_init(&S.w_empty[b], p.nr == 32 ? NEPI / 2 : NEPI);
      mbar_init(&S.x_full[b], 1);
      mbar_init(&S.x_empty[b], NEPI);
    }
    mbar_init(&S.dz1p_full, 1);
    mbar_init(&S.dz1p_empty, NEPI);
    mbar_init(&S.dz1_full, NEPI);
    mbar_init(&S.fin, 1);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(&S.tmem_base);
  pdl_wait();  // nothing a previous grid writes is touched before this point
  pdl_trigger();
  if (threadIdx.x < RP) {
    S.Dc1[threadIdx.x] = p.Dc1[threadIdx.x];
    S.Dc2[threadIdx.x] = p.Dc2[threadIdx.x];
  }
  zero_list(p.zero);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;
  const int nitems = p.nM + p.nH + p.nN;
  if (threadIdx.x == 0) TL_STAMP(1, 0);

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int it = 0, tl = 0;
      int last_parity[FFN_NST_B];
      for (int s = 0; s < FFN_NST_B; ++s) last_parity[s] = -1;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x, ++tl) {
        const int tok0 = tile * TILE;
        // the two rank tiles are free once the previous tile's phase C is done
        if (!wait_bar(&S.zt_empty, (tl & 1) ^ 1, abort_flag, 70)) break;
        mbar_expect_tx(&S.zl_full, 2 * BOX);
        tma_load(zt1, &tm_zs1, &S.zl_full, 0, tok0);
        tma_load(zt2, &tm_zs2, &S.zl_full, 0, tok0);
        for (int c = 0; c < nitems; ++c, ++it) {
          const int s = it % FFN_NST_B;
          const uint32_t ph = (it / FFN_NST_B) & 1;
          if (!wait_bar(&S.empty[s], ph ^ 1, abort_flag, 71)) { ok = false; break; }
          uint8_t* st = stages + s * STAGE;
          if (c < p.nM) {
            const int col = rot_chunk(c, p.nM, tile) * CH;
            mbar_expect_tx(&S.full[s], 3 * BOX);
            tma_load(st, &tm_dy, &S.full[s], col, tok0);
            tma_load(st + BOX, &tm_dy, &S.full[s], col + 64, tok0);
            tma_load(st + OPND, &tm_bm2, &S.full[s], col, 0);
            tma_load(st + OPND + BOX / 2, &tm_bm2, &S.full[s], col + 64, 0);
          } else if (c < p.nM + p.nH) {
            const int col = rot_chunk(c - p.nM, p.nH, tile) * CH;
            mbar_expect_tx(&S.full[s], 2 * BOX);
            tma_load(st, &tm_anr2, &S.full[s], 0, col);
            tma_load(st + OPND, &tm_bm1, &S.full[s], col, 0);
            tma_load(st + OPND + BOX / 2, &tm_bm1, &S.full[s], col + 64, 0);
          } else {
            const int col = rot_chunk(c - p.nM - p.nH, p.nN, tile) * CH;
            mbar_expect_tx(&S.full[s], 3 * BOX);
            tma_load(st, &tm_x, &S.full[s], col, tok0);
            tma_load(st + BOX, &tm_x, &S.full[s], col + 64, tok0);
            tma_load(st + OPND, &tm_anr1, &S.full[s], 0, col);
          }
          last_parity[s] = (int)ph;
        }
      }
      for (int s = 0; s < FFN_NST_B; ++s)
        if (last_parity[s] >= 0) drain_bar(&S.full[s], (uint32_t)last_parity[s]);
      if (tl > 0) drain_bar(&S.zl_full, (uint32_t)((tl - 1) & 1));
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_r = idesc(128, p.nr, 0, 0);  // token x rank, both K-major
      const uint32_t id_w = idesc(128, p.nr, 1, 1);  // weight x rank, both MN-major
      const uint32_t id_n = idesc(128, 128, 0, 0);   // token x 128 columns, K = rank
      const uint32_t id_h = idesc(128, 128, 0, 1);   // token x 128 columns, B MN-major
      const uint32_t z1a = su32(zt1), z2a = su32(zt2);
      const uint32_t ata = su32(atile), dha = su32(dhtile);
      int it = 0, wc = 0, xc = 0, hdc = 0, adc = 0, tl = 0;
      bool ok = true;
      // the W buffer for the next weight-side product (waits for its drain)
      auto w_take = [&](uint32_t& col) -> bool {
        const int wb = wc & 1;
        if (!wait_bar(&S.w_empty[wb], ((wc >> 1) & 1) ^ 1, abort_flag, 72)) return false;
        tc_fence_after();
        col = tmem + FB_W + wb * 64;
        return true;
      };
      auto w_done = [&]() {
        mma_commit(&S.w_full[wc & 1]);
        ++wc;
      };
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x, ++tl) {
        if (!wait_bar(&S.zl_full, tl & 1, abort_flag, 73)) break;
        // B: dz2' = dy B2^T ; dB2^T chunk = dy^T z2'
        if (!wait_bar(&S.dzp2_empty, (tl & 1) ^ 1, abort_flag, 74)) break;
        tc_fence_after();
        for (int c = 0; c < p.nM; ++c, ++it) {
          const int s = it % FFN_NST_B;
          if (!wait_bar(&S.full[s], (it / FFN_NST_B) & 1, abort_flag, 75)) { ok = false; break; }
          if (tl == 0 && c < 6) TLW(1, 24 + c);
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma(tmem + FB_DZ2P, kdesc(st + b * BOX) + 2 * k,
                  kdesc(st + OPND + b * (BOX / 2)) + 2 * k, id_r, (c | b | k) != 0);
          uint32_t wcol;
          if (!w_take(wcol)) { ok = false; break; }
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma(wcol, mndesc(st, BOX) + 128 * k, mndesc(z2a, 1024) + 128 * k, id_w, k != 0);
          w_done();
          mma_commit(&S.empty[s]);
        }
        if (!ok) break;
        mma_commit(&S.dzp2_full);
        mma_commit(&S.zp2_free);
        if (tl == 0) TLW(1, 30);
        // hidden chunks
        if (!wait_bar(&S.dz2_full, tl & 1, abort_flag, 76)) break;
        if (tl == 0) TLW(1, 31);
        if (!wait_bar(&S.dz1p_empty, (tl & 1) ^ 1, abort_flag, 77)) break;
        tc_fence_after();
        const int ih = it;
        // h_c = z1' B1[:, c] and da_c = dz2 A2[c, :]^T into the single H / DA pair
        auto issue_hd = [&](int c) -> bool {
          const int s = (ih + c) % FFN_NST_B;
          if (!wait_bar(&S.full[s], ((ih + c) / FFN_NST_B) & 1, abort_flag, 78)) return false;
          if (tl == 0 && c < 4) TLW(1, 16 + c);
          if (tl == 0 && c >= 4 && c < 8) TLW(1, 32 + 3 * (c - 4));
          if (!wait_bar(&S.hd_empty, (hdc & 1) ^ 1, abort_flag, 79)) return false;
          if (tl == 0 && c < 4) TLW(1, 20 + c);
          if (tl == 0 && c >= 4 && c < 8) TLW(1, 33 + 3 * (c - 4));
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
          for (int k = 0; k < p.kb1; ++k)
            mma(tmem + FB_H, kdesc(z1a) + 2 * k, mndesc(st + OPND, BOX / 2) + 128 * k, id_h, k != 0);
          for (int k = 0; k < p.kb2; ++k)
            mma(tmem + FB_DA, kdesc(z2a) + 2 * k, kdesc(st) + 2 * k, id_n, k != 0);
          mma_commit(&S.hd_full);
          if (tl == 0 && c < 8) TLW(1, 2 * c);
          ++hdc;
          return true;
        };
        if (!issue_hd(0)) break;
        for (int c = 0; c < p.nH; ++c) {
          if (c + 1 < p.nH && !issue_hd(c + 1)) { ok = false; break; }
          if (!wait_bar(&S.ad_full, adc & 1, abort_flag, 80)) { ok = false; break; }
          if (tl == 0 && c < 8) TLW(1, 2 * c + 1);
          tc_fence_after();
          const int s = (ih + c) % FFN_NST_B;
          const uint32_t st = su32(stages + s * STAGE);
#pragma unroll
          for (int b = 0; b < 2; ++b)   // dz1' += dh_c B1[:, c]^T
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma(tmem + FB_DZ1P, kdesc(dha + b * BOX) + 2 * k,
                  kdesc(st + OPND + b * (BOX / 2)) + 2 * k, id_r, (c | b | k) != 0);
          uint32_t wcol;
          if (!w_take(wcol)) { ok = false; break; }
#pragma unroll
          for (int k = 0; k < 8; ++k)   // dA2 chunk = a_c^T dz2
            mma(wcol, mndesc(ata, BOX) + 128 * k, mndesc(z2a, 1024) + 128 * k, id_w, k != 0);
          w_done();
          if (!w_take(wcol)) { ok = false; break; }
#pragma unroll
          for (int k = 0; k < 8; ++k)   // dB1^T chunk = dh_c^T z1'
            mma(wcol, mndesc(dha, BOX) + 128 * k, mndesc(z1a, 1024) + 128 * k, id_w, k != 0);
          w_done();
          mma_commit(&S.ad_empty);
          mma_commit(&S.empty[s]);
          if (tl == 0 && c >= 4 && c < 8) TLW(1, 34 + 3 * (c - 4));
          ++adc;
        }
        if (!ok) break;
        it = ih + p.nH;
        mma_commit(&S.dz1p_full);
        // C: dx = dz1 A1^T ; dA1 chunk = x^T dz1
        if (!wait_bar(&S.dz1_full, tl & 1, abort_flag, 81)) break;
        tc_fence_after();
        for (int c = 0; c < p.nN; ++c, ++it, ++xc) {
          const int s = it % FFN_NST_B;
          const int xb = xc & 1;
          if (!wait_bar(&S.full[s], (it / FFN_NST_B) & 1, abort_flag, 82)) { ok = false; break; }
          if (!wait_bar(&S.x_empty[xb], ((xc >> 1) & 1) ^ 1, abort_flag, 83)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
          for (int k = 0; k < p.kb1; ++k)
            mma(tmem + FB_X + xb * 128, kdesc(z1a) + 2 * k, kdesc(st + OPND) + 2 * k, id_n, k != 0);
          mma_commit(&S.x_full[xb]);
          uint32_t wcol;
          if (!w_take(wcol)) { ok = false; break; }
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma(wcol, mndesc(st, BOX) + 128 * k, mndesc(z1a, 1024) + 128 * k, id_w, k != 0);
          w_done();
          mma_commit(&S.empty[s]);
        }
        if (!ok) break;
        mma_commit(&S.zt_empty);
      }
      mma_commit(&S.fin);
      drain_bar(&S.fin, 0);
    }
  } else {
    // ---------------- epilogue: 8 warps, thread = (token row, column half)
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int row = 32 * q + lane;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const int r1 = p.rinfo1[0], r2 = p.rinfo2[0];
    uint8_t* box = staging + (warp - 2) * STG;
    int wc = 0, xc = 0, hdc = 0, adc = 0, tl = 0;
    // drain the next W buffer: 32 rank columns of 32 weight rows, bulk-added
    // into the token sum `map` at (row0 + 32 q, col0) when row0 + 32 q < nrows.
    // 64 rank columns: every warp drains every buffer, half h its columns 32 h..;
    // 32 rank columns: buffer b is drained by the warps of half b alone, so the
    // two W products of a hidden chunk are drained side by side
    auto drain_w = [&](const CUtensorMap* map, int row0, int nrows, int rprime) -> bool {
      float v[32];
      const int wb = wc & 1;
      const int col0 = p.nr == 32 ? 0 : 32 * h;
      if (p.nr == 32 && wb != h) {
        ++wc;
        return true;
      }
      if (!warp_wait(&S.w_full[wb], (wc >> 1) & 1, abort_flag, 84)) return false;
      tc_fence_after();
      tmem_ld32(tmem + lane_off + FB_W + wb * 64 + col0, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.w_empty[wb]);
      ++wc;
      if (col0 < rprime && row0 + 32 * q < nrows) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        stage_f32_32(box, lane, v);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int r = (p.det ? (int)blockIdx.x * nrows : 0) + row0 + 32 * q;
          if (p.det && tl == 0)
            tma_store(map, box, col0, r);
          else
            tma_reduce_add(map, box, col0, r);
          bulk_commit();
        }
      }
      return true;
    };
    // column sums over this warp's 32 rows of z' dz' / Dc: the token sum of z dz'
    auto dd_sum = [&](const float (&z)[32], const float (&v)[32], const float* Dc, float* out,
                      float* slot, int rprime) {
      float pr[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) pr[j] = z[j] * v[j];
      const float colsum = warp_transpose_sum(pr, lane);
      if (32 * h + lane < rprime) {
        const float d = colsum / Dc[32 * h + lane];
        if (p.det) {  // this lane alone owns the entry of its CTA and quadrant
          float* e = slot + ((size_t)blockIdx.x * 4 + q) * RP + 32 * h + lane;
          *e = tl == 0 ? d : *e + d;
        } else {
          atomicAdd(out + 32 * h + lane, d);
        }
      }
    };
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++tl) {
      float z[32], v[32];
      bool ok = true;
      // E1: dB2^T chunks
      for (int c = 0; c < p.nM; ++c)
        if (!drain_w(&tm_dbc2, rot_chunk(c, p.nM, tile) * CH, p.M, r2)) { ok = false; break; }
      if (!ok) break;
      // E2: dz2' -> dD2, dz2 tile (over z2', whose readers are done)
      if (!warp_wait(&S.dzp2_full, tl & 1, abort_flag, 85)) break;
      if (warp == 2 && lane == 0 && tl == 0) TL_STAMP(1, 1);
      tc_fence_after();
      if (32 * h < p.nr) {
        tmem_ld32(tmem + lane_off + FB_DZ2P + 32 * h, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;  // rank columns the MMAs left out
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.dzp2_empty);
      if (!warp_wait(&S.zl_full, tl & 1, abort_flag, 86)) break;
      ld_tile_half(zt2, row, h, z);
      dd_sum(z, v, S.Dc2, p.dDc2, p.dDslot2, r2);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= S.Dc2[32 * h + j];
      if (!warp_wait(&S.zp2_free, tl & 1, abort_flag, 87)) break;
      __syncwarp();  // every lane has read its z2' row before any lane overwrites it
      st_tile_half(zt2, row, h, v);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.dz2_full);
      // E3: hidden chunks
      for (int c = 0; c < p.nH; ++c) {
        float h0[32], h1[32], d0[32], d1[32];
        if (!warp_wait(&S.hd_full, hdc & 1, abort_flag, 88)) { ok = false; break; }
        if (warp == 2 && lane == 0 && tl == 0 && c < 3) TL_STAMP(1, 2 + 3 * c);
        if (tl == 0 && c < 8) TLW(1, 4 * c);
        tc_fence_after();
        tmem_ld32(tmem + lane_off + FB_H + 64 * h, h0);
        tmem_ld32(tmem + lane_off + FB_H + 64 * h + 32, h1);
        tmem_ld32(tmem + lane_off + FB_DA + 64 * h, d0);
        tmem_ld32(tmem + lane_off + FB_DA + 64 * h + 32, d1);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.hd_empty);
        ++hdc;
        uint32_t pa0[16], pa1[16], pd0[16], pd1[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float2 a, g;
          gelu_tanh_grad2(make_float2(h0[2 * j], h0[2 * j + 1]),
                          make_float2(d0[2 * j], d0[2 * j + 1]), a, g);
          pa0[j] = pack_bf16(a.x, a.y);
          pd0[j] = pack_bf16(g.x, g.y);
          gelu_tanh_grad2(make_float2(h1[2 * j], h1[2 * j + 1]),
                          make_float2(d1[2 * j], d1[2 * j + 1]), a, g);
          pa1[j] = pack_bf16(a.x, a.y);
          pd1[j] = pack_bf16(g.x, g.y);
        }
        if (warp == 2 && lane == 0 && tl == 0 && c < 3) TL_STAMP(1, 3 + 3 * c);
        if (tl == 0 && c < 8) TLW(1, 4 * c + 1);
        if (!warp_wait(&S.ad_empty, (adc & 1) ^ 1, abort_flag, 89)) { ok = false; break; }
        if (warp == 2 && lane == 0 && tl == 0 && c < 3) TL_STAMP(1, 4 + 3 * c);
        if (tl == 0 && c < 8) TLW(1, 4 * c + 2);
        st_tile_half_u(atile + h * BOX, row, 0, pa0);
        st_tile_half_u(atile + h * BOX, row, 1, pa1);
        st_tile_half_u(dhtile + h * BOX, row, 0, pd0);
        st_tile_half_u(dhtile + h * BOX, row, 1, pd1);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.ad_full);
        if (tl == 0 && c < 8) TLW(1, 4 * c + 3);
        ++adc;
        if (c > 0) {  // the previous chunk's dA2 and dB1^T products
          const int cb = rot_chunk(c - 1, p.nH, tile) * CH;
          if (!drain_w(&tm_dac2, cb, p.H, r2) || !drain_w(&tm_dbc1, cb, p.H, r1)) {
            ok = false;
            break;
          }
        }
        if (tl == 0 && c < 8) TLW(1, 32 + c);
      }
      if (!ok) break;
      {
        const int cb = rot_chunk(p.nH - 1, p.nH, tile) * CH;
        if (!drain_w(&tm_dac2, cb, p.H, r2) || !drain_w(&tm_dbc1, cb, p.H, r1)) break;
      }
      // E4: dz1' -> dD1, dz1 tile (over z1', whose readers are done)
      if (!warp_wait(&S.dz1p_full, tl & 1, abort_flag, 90)) break;
      if (warp == 2 && lane == 0 && tl == 0) TL_STAMP(1, 11);
      tc_fence_after();
      if (32 * h < p.nr) {
        tmem_ld32(tmem + lane_off + FB_DZ1P + 32 * h, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.dz1p_empty);
      ld_tile_half(zt1, row, h, z);
      dd_sum(z, v, S.Dc1, p.dDc1, p.dDslot1, r1);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= S.Dc1[32 * h + j];
      __syncwarp();
      st_tile_half(zt1, row, h, v);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.dz1_full);
      // E5: dx chunks and dA1 chunks
      for (int c = 0; c < p.nN; ++c, ++xc) {
        const int xb = xc & 1;
        if (!warp_wait(&S.x_full[xb], (xc >> 1) & 1, abort_flag, 91)) { ok = false; break; }
        tc_fence_after();
        const int cx = rot_chunk(c, p.nN, tile);
        const int col = cx * CH + 64 * h;
        const bool st_dx = col < p.N && (int64_t)tile * TILE + 32 * q < p.T;
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {
          tmem_ld32(tmem + lane_off + FB_X + xb * 128 + 64 * h + 32 * piece, v);
          stage_bf16_32(box, lane, piece, v);
        }
        tc_fence_before();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&S.x_empty[xb]);
          if (st_dx) {
            tma_store(&tm_dx, box, col, tile * TILE + 32 * q);
            bulk_commit();
          }
        }
        if (!drain_w(&tm_dac1, cx * CH, p.N, r1)) { ok = false; break; }
      }
      if (!ok) break;
      if (warp == 2 && lane == 0 && tl == 0) TL_STAMP(1, 12);
      // the next tile's adds into this CTA's slots come after this tile's
      if (p.det && lane == 0) bulk_wait_all();
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) TL_STAMP(1, 13);
  if (warp == 1) tmem_free(tmem);
}

cudaError_t set_ffn_attrs() {
  static PerDevice once;
  return once.get([] {
    cudaError_t e = cudaFuncSetAttribute(ffn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemFfnFwd);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ffn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemFfnBwd);
    return e;
  });
}

// 16-wide K blocks that cover a middle rank (ranks past it are zero padding)
int kblocks(int rd) { return (rd < RP ? rd : RP) + 15 >> 4; }

}  // namespace

bool ffn_tc_supported(const LayerPlan& U, const LayerPlan& D) {
  return tc_supported(U) && tc_supported(D) && U.M == D.N;
}

tt_status ffn_tc_forward(const LayerPlan& U, const LayerPlan& D, int64_t T, const void* x, void* y,
                         void* ws, size_t off1, size_t off2, void* zs1, void* zs2,
                         bool prefetch_x, cudaStream_t st) {
  if (T <= 0) return TT_OK;
  if (T > (int64_t)0x7FFFFFFF - TILE || !ffn_tc_supported(U, D)) return TT_ERR_UNSUPPORTED;
  if (!y && (!zs1 || !zs2)) return TT_ERR_INVALID_ARG;
  if (set_ffn_attrs() != cudaSuccess) return TT_ERR_CUDA;
  const TcLayout t1 = tc_layout(U), t2 = tc_layout(D);
  void* anr1 = at<void>(ws, off1 + t1.Anr);
  void* bm1 = at<void>(ws, off1 + t1.Bm);
  void* anr2 = at<void>(ws, off2 + t2.Anr);
  void* bm2 = at<void>(ws, off2 + t2.Bm);
  void* any = y ? y : zs1;
  CUtensorMap mx, manr1, mbm1, manr2, mbm2, my, mzs1, mzs2;
  if (!make_map(&mx, x, U.N, T, 64, TILE) || !make_map(&manr1, anr1, RP, U.N, 64, CH) ||
      !make_map(&mbm1, bm1, U.M, RP, 64, RP) || !make_map(&manr2, anr2, RP, D.N, 64, CH) ||
      !make_map(&mbm2, bm2, D.M, RP, 64, RP) ||
      !make_map(&my, y ? y : any, y ? D.M : RP, T, 64, 32) ||
      !make_map(&mzs1, zs1 ? zs1 : any, RP, T, 64, TILE) ||
      !make_map(&mzs2, zs2 ? zs2 : any, RP, T, 64, TILE))
    return TT_ERR_CUDA;
  FfnFwdArgs a;
  a.T = T;
  a.nN = (int)((U.N + CH - 1) / CH);
  a.nH = (int)((U.M + CH - 1) / CH);
  a.nM = y ? (int)((D.M + CH - 1) / CH) : 0;  // no y: the kept z1', z2' only
  a.ntiles = (int)((T + TILE - 1) / TILE);
  a.kb1 = kblocks(U.rd);
  a.kb2 = kblocks(D.rd);
  a.nr = U.rd <= 32 && D.rd <= 32 ? 32 : 64;
  a.save_z = (zs1 && zs2) ? 1 : 0;
  a.M = (int)D.M;
  a.prefetch_x = prefetch_x && pdl_enabled() ? 1 : 0;
  a.Dc1 = at<float>(ws, off1 + t1.Dc);
  a.Dc2 = at<float>(ws, off2 + t2.Dc);
  const int grid = a.ntiles < num_sms() ? a.ntiles : num_sms();
  cudaError_t e = launch_ex(ffn_fwd_kernel, grid, NTHREADS, kSmemFfnFwd, st, false, mx, manr1,
                            mbm1, manr2, mbm2, my, mzs1, mzs2, a);
  count_launches(1);
  return e == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

tt_status ffn_tc_backward(const LayerPlan& U, const LayerPlan& D, int64_t T, const void* x,
                          const void* dy, void* dx, void* ws, size_t off1, size_t off2,
                          const void* zs1, const void* zs2, const ZeroList& zero,
                          const DetSlots* det1, const DetSlots* det2, cudaStream_t st) {
  if (!ffn_tc_supported(U, D)) return TT_ERR_UNSUPPORTED;
  if (T <= 0) return zero_list_memset(zero, st) == cudaSuccess ? TT_OK : TT_ERR_CUDA;
  if (T > (int64_t)0x7FFFFFFF - TILE) return TT_ERR_UNSUPPORTED;
  if ((det1 == nullptr) != (det2 == nullptr)) return TT_ERR_INVALID_ARG;
  const bool det = det1 != nullptr;
  if (det && (det1->count < 1 || det2->count != det1->count ||
              (int64_t)det1->count * (U.M > U.N ? U.M : U.N) > 0x7FFFFFFF ||
              (int64_t)det1->count * (D.M > D.N ? D.M : D.N) > 0x7FFFFFFF))
    return TT_ERR_UNSUPPORTED;
  const int64_t nslot = det ? det1->count : 1;
  if (set_ffn_attrs() != cudaSuccess) return TT_ERR_CUDA;
  const TcLayout t1 = tc_layout(U), t2 = tc_layout(D);
  CUtensorMap mx, mdy, manr1, mbm1, manr2, mbm2, mdx, mdac1, mdbc1, mdac2, mdbc2, mzs1, mzs2;
  if (!make_map(&mx, x, U.N, T, 64, TILE) || !make_map(&mdy, dy, D.M, T, 64, TILE) ||
      !make_map(&manr1, at<void>(ws, off1 + t1.Anr), RP, U.N, 64, CH) ||
      !make_map(&mbm1, at<void>(ws, off1 + t1.Bm), U.M, RP, 64, RP) ||
      !make_map(&manr2, at<void>(ws, off2 + t2.Anr), RP, D.N, 64, CH) ||
      !make_map(&mbm2, at<void>(ws, off2 + t2.Bm), D.M, RP, 64, RP) ||
      !make_map(&mdx, dx, U.N, T, 64, 32) ||
      !make_map(&mdac1, det ? det1->a : at<void>(ws, off1 + t1.dAc), RP, U.N * nslot, 32, 32,
                kMapF32) ||
      !make_map(&mdbc1, det ? det1->b : at<void>(ws, off1 + t1.dBc), RP, U.M * nslot, 32, 32,
                kMapF32) ||
      !make_map(&mdac2, det ? det2->a : at<void>(ws, off2 + t2.dAc), RP, D.N * nslot, 32, 32,
                kMapF32) ||
      !make_map(&mdbc2, det ? det2->b : at<void>(ws, off2 + t2.dBc), RP, D.M * nslot, 32, 32,
                kMapF32) ||
      !make_map(&mzs1, zs1, RP, T, 64, TILE) || !make_map(&mzs2, zs2, RP, T, 64, TILE))
    return TT_ERR_CUDA;
  FfnBwdArgs a;
  a.T = T;
  a.nN = (int)((U.N + CH - 1) / CH);
  a.nH = (int)((U.M + CH - 1) / CH);
  a.nM = (int)((D.M + CH - 1) / CH);
  a.ntiles = (int)((T + TILE - 1) / TILE);
  a.kb1 = kblocks(U.rd);
  a.kb2 = kblocks(D.rd);
  // (a deterministic pass keeps every W drain on the same warp from tile to
  // tile: the 64-wide products, whose drains split by column half)
  a.nr = !det && U.rd <= 32 && D.rd <= 32 ? 32 : 64;
  a.N = (int)U.N;
  a.H = (int)U.M;
  a.M = (int)D.M;
  a.Dc1 = at<float>(ws, off1 + t1.Dc);
  a.Dc2 = at<float>(ws, off2 + t2.Dc);
  a.rinfo1 = at<int>(ws, off1 + t1.rinfo);
  a.rinfo2 = at<int>(ws, off2 + t2.rinfo);
  a.dDc1 = at<float>(ws, off1 + t1.dDc);
  a.dDc2 = at<float>(ws, off2 + t2.dDc);
  a.zero = zero;
  a.det = det ? 1 : 0;
  a.dDslot1 = det ? det1->d : nullptr;
  a.dDslot2 = det ? det2->d : nullptr;
  int grid = a.ntiles < num_sms() ? a.ntiles : num_sms();
  if (det && grid > det1->count) grid = det1->count;
  cudaError_t e = launch_ex(ffn_bwd_kernel, grid, NTHREADS, kSmemFfnBwd, st, false, mx, mdy,
                            manr1, mbm1, manr2, mbm2, mdx, mdac1, mdbc1, mdac2, mdbc2, mzs1, mzs2,
                            a);
  count_launches(1);
  if (e != cudaSuccess) return TT_ERR_CUDA;
  if (det) {  // each layer's slots of the `grid` CTAs, summed in CTA order
    e = det_sum_launch(U, *det1, grid, at<float>(ws, off1 + t1.dAc), at<float>(ws, off1 + t1.dBc),
                       a.dDc1, st);
    if (e == cudaSuccess)
      e = det_sum_launch(D, *det2, grid, at<float>(ws, off2 + t2.dAc),
                         at<float>(ws, off2 + t2.dBc), a.dDc2, st);
    if (e != cudaSuccess) return TT_ERR_CUDA;
  }
  return TT_OK;
}

}  // namespace ttc

extern "C" tt_status tt_gelu_rate(int mode, int iters, int blocks, float* out, void* stream) {
  if ((mode != 0 && mode != 1) || iters < 1 || blocks < 1 || !out) return TT_ERR_INVALID_ARG;
  ttc::gelu_rate_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(mode, iters, out);
  ttc::count_launches(1);
  return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

#ifdef TTC_TIMELINE
extern "C" int ttc_timeline_warps_read(void* host, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(host, ttc::g_tlw, bytes);
}
#endif
