// Several TT layers that read the same input (the Q, K and V projections of
// an attention block): one kernel per pass streams x once for all of them.
// Included once, by tc_fused.cu, after the single-layer kernels (it uses
// their PTX helpers and the per-device status word).
//
// Forward, per tile of 128 tokens and G <= 3 layers g:
//   z_g = x A_g for every g in one pass over x (TMEM, 64 columns each)
//   for each g: z'_g = z_g diag(D_g) -> bf16 tile; y_g = z'_g B_g
// Backward, with the forward's z'_g tiles:
//   for each g: dz'_g = dy_g B_g^T ; dB_g^T += dy_g^T z'_g ; dD_g += sum z_g dz'_g
//   one pass over x: dx = sum_g dz_g A_g^T ; dA_g += x^T dz_g for every g
// The activations (x, dy_g) and the per-layer operands (A_g rows, B_g
// columns) come through two TMA rings, so that one x chunk serves G operand
// chunks.
#pragma once

namespace ttc {
namespace {

constexpr int kMaxGroups = 3;
constexpr int QKV_NACT = 2;   // activation ring: [128 tokens][128 columns] bf16 (two boxes)
constexpr int QKV_NOP = 3;    // operand ring: one 16 KB operand chunk each
constexpr int ACT_STAGE = 2 * BOX;

struct QkvFwdArgs {
  int64_t T;
  int G, nN, ntiles, tt;  // tt: tokens a tile (a multiple of 16, at most 128)
  int nM[kMaxGroups];
  int M[kMaxGroups];
  int kb[kMaxGroups];
  int save_z;
  int prefetch_x;  // x of the first chunks requested before the dependency wait
  const float* Dc[kMaxGroups];
};

// Zero rows [tt, TILE) of n activation boxes (contiguous from `boxes`) and
// of m more boxes from `more`: the loads of a tt-row tile leave them alone,
// and the MMAs read all 128 rows.
__device__ void zero_tail_boxes(uint8_t* boxes, int n, uint8_t* more, int m, int tt) {
  if (tt >= TILE) return;
  const int per_box = (TILE - tt) * 8;  // 16-byte units
  for (int i = threadIdx.x; i < (n + m) * per_box; i += blockDim.x) {
    const int b = i / per_box, o = i - b * per_box;
    uint8_t* bp = b < n ? boxes + b * BOX : more + (b - n) * BOX;
    *reinterpret_cast<uint4*>(bp + tt * 128 + o * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_async_smem();
}

struct QkvSmem {
  uint64_t a_full[QKV_NACT], a_empty[QKV_NACT];
  uint64_t o_full[QKV_NOP], o_empty[QKV_NOP];
  uint64_t z_full, z_empty, zp_full, zp_empty;
  uint64_t x_full[2], x_empty[2];
  uint64_t w_full[2], w_empty[2];
  uint64_t zl_full, zt_empty, dzp_full, dzp_empty, dz_full, fin;
  uint32_t tmem_base;
  int abort_flag;
  float Dc[kMaxGroups][RP];
};

// TMEM columns of the forward: z_g at 64 g, y double buffer at 192
constexpr uint32_t QF_Z = 0, QF_Y = 192;

constexpr size_t kSmemQkvFwd =
    QKV_NACT * ACT_STAGE + QKV_NOP * BOX + BOX + NEPI * 2 * STG + sizeof(QkvSmem) + 1024;
static_assert(kSmemQkvFwd <= 227 * 1024, "QKV forward smem");

__global__ void __launch_bounds__(NTHREADS, 1)
    qkv_fwd_kernel(const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_anr0,
                   const __grid_constant__ CUtensorMap tm_anr1,
                   const __grid_constant__ CUtensorMap tm_anr2,
                   const __grid_constant__ CUtensorMap tm_bm0,
                   const __grid_constant__ CUtensorMap tm_bm1,
                   const __grid_constant__ CUtensorMap tm_bm2,
                   const __grid_constant__ CUtensorMap tm_y0,
                   const __grid_constant__ CUtensorMap tm_y1,
                   const __grid_constant__ CUtensorMap tm_y2,
                   const __grid_constant__ CUtensorMap tm_y16_0,
                   const __grid_constant__ CUtensorMap tm_y16_1,
                   const __grid_constant__ CUtensorMap tm_y16_2,
                   const __grid_constant__ CUtensorMap tm_zs0,
                   const __grid_constant__ CUtensorMap tm_zs1,
                   const __grid_constant__ CUtensorMap tm_zs2, QkvFwdArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1k(smem_raw);
  uint8_t* act = base;                              // activation ring
  uint8_t* opr = act + QKV_NACT * ACT_STAGE;        // operand ring
  uint8_t* zp_tile = opr + QKV_NOP * BOX;           // z'_g, one layer at a time
  uint8_t* staging = zp_tile + BOX;                 // 2 boxes per epilogue warp
  QkvSmem& S = *reinterpret_cast<QkvSmem*>(staging + NEPI * 2 * STG);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const CUtensorMap* tm_anr[kMaxGroups] = {&tm_anr0, &tm_anr1, &tm_anr2};
  const CUtensorMap* tm_bm[kMaxGroups] = {&tm_bm0, &tm_bm1, &tm_bm2};
  const CUtensorMap* tm_y[kMaxGroups] = {&tm_y0, &tm_y1, &tm_y2};
  const CUtensorMap* tm_y16[kMaxGroups] = {&tm_y16_0, &tm_y16_1, &tm_y16_2};
  const CUtensorMap* tm_zs[kMaxGroups] = {&tm_zs0, &tm_zs1, &tm_zs2};

  if (threadIdx.x == 0) {
    for (int s = 0; s < QKV_NACT; ++s) {
      mbar_init(&S.a_full[s], 1);
      mbar_init(&S.a_empty[s], 1);
    }
    for (int s = 0; s < QKV_NOP; ++s) {
      mbar_init(&S.o_full[s], 1);
      mbar_init(&S.o_empty[s], 1);
    }
    mbar_init(&S.z_full, 1);
    mbar_init(&S.z_empty, NEPI);
    mbar_init(&S.zp_full, NEPI);
    mbar_init(&S.zp_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.x_full[b], 1);
      mbar_init(&S.x_empty[b], NEPI);
    }
    mbar_init(&S.fin, 1);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int s = 0; s < fwd_prefetched(p, QKV_NACT); ++s) {  // x of the first chunks
      uint8_t* st = act + s * ACT_STAGE;
      mbar_expect_tx(&S.a_full[s], 2 * (uint32_t)p.tt * 128);
      tma_load(st, &tm_x, &S.a_full[s], s * CH, blockIdx.x * p.tt);
      tma_load(st + BOX, &tm_x, &S.a_full[s], s * CH + 64, blockIdx.x * p.tt);
    }
  }
  if (warp == 1) tmem_alloc(&S.tmem_base);
  pdl_wait();  // nothing a previous grid writes is touched before this point (but x above)
  pdl_trigger();
  for (int i = threadIdx.x; i < p.G * RP; i += blockDim.x) S.Dc[i / RP][i % RP] = p.Dc[i / RP][i % RP];
  zero_tail_boxes(act, 2 * QKV_NACT, zp_tile, 1, p.tt);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;

  if (warp == 0) {
    // ---------------- TMA producer: x chunks (activation ring) with every
    // layer's A rows (operand ring), then every layer's B columns
    if (lane == 0) {
      int ia = 0, io = 0;
      int lpa[QKV_NACT], lpo[QKV_NOP];
      for (int s = 0; s < QKV_NACT; ++s) lpa[s] = -1;
      for (int s = 0; s < QKV_NOP; ++s) lpo[s] = -1;
      bool ok = true;
      auto take_op = [&](int& s) -> bool {
        s = io % QKV_NOP;
        const uint32_t ph = (io / QKV_NOP) & 1;
        if (!wait_bar(&S.o_empty[s], ph ^ 1, abort_flag, 120)) return false;
        lpo[s] = (int)ph;
        ++io;
        return true;
      };
      const uint32_t act_bytes = (uint32_t)p.tt * 128;  // one activation box of tt rows
      const int npre = fwd_prefetched(p, QKV_NACT);     // x already requested
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x) {
        const int tok0 = tile * p.tt;
        for (int c = 0; ok && c < p.nN; ++c) {
          const int s = ia % QKV_NACT;
          const uint32_t ph = (ia / QKV_NACT) & 1;
          if (!wait_bar(&S.a_empty[s], ph ^ 1, abort_flag, 121)) { ok = false; break; }
          uint8_t* st = act + s * ACT_STAGE;
          if (ia >= npre) {
            mbar_expect_tx(&S.a_full[s], 2 * act_bytes);
            tma_load(st, &tm_x, &S.a_full[s], c * CH, tok0);
            tma_load(st + BOX, &tm_x, &S.a_full[s], c * CH + 64, tok0);
          }
          lpa[s] = (int)ph;
          ++ia;
          for (int g = 0; g < p.G; ++g) {
            int so;
            if (!take_op(so)) { ok = false; break; }
            mbar_expect_tx(&S.o_full[so], BOX);
            tma_load(opr + so * BOX, tm_anr[g], &S.o_full[so], 0, c * CH);
          }
        }
        for (int g = 0; ok && g < p.G; ++g)
          for (int c = 0; c < p.nM[g]; ++c) {
            int so;
            if (!take_op(so)) { ok = false; break; }
            mbar_expect_tx(&S.o_full[so], BOX);
            tma_load(opr + so * BOX, tm_bm[g], &S.o_full[so], c * CH, 0);
            tma_load(opr + so * BOX + BOX / 2, tm_bm[g], &S.o_full[so], c * CH + 64, 0);
          }
      }
      for (int s = 0; s < QKV_NACT; ++s)
        if (lpa[s] >= 0) drain_bar(&S.a_full[s], (uint32_t)lpa[s]);
      for (int s = 0; s < QKV_NOP; ++s)
        if (lpo[s] >= 0) drain_bar(&S.o_full[s], (uint32_t)lpo[s]);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_z = idesc(128, 64, 0, 1);   // B = A_g rows, MN-major
      const uint32_t id_y = idesc(128, 128, 0, 1);  // B = B_g columns, MN-major
      const uint32_t zp_addr = su32(zp_tile);
      int ia = 0, io = 0, yc = 0, tl = 0, zu = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x, ++tl) {
        if (!wait_bar(&S.z_empty, (tl & 1) ^ 1, abort_flag, 122)) break;
        tc_fence_after();
        for (int c = 0; c < p.nN; ++c, ++ia) {
          const int s = ia % QKV_NACT;
          if (!wait_bar(&S.a_full[s], (ia / QKV_NACT) & 1, abort_flag, 123)) { ok = false; break; }
          const uint32_t st = su32(act + s * ACT_STAGE);
          for (int g = 0; g < p.G; ++g, ++io) {
            const int so = io % QKV_NOP;
            if (!wait_bar(&S.o_full[so], (io / QKV_NOP) & 1, abort_flag, 124)) { ok = false; break; }
            tc_fence_after();
            const uint32_t ob = su32(opr + so * BOX);
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma(tmem + QF_Z + 64 * g, kdesc(st + b * BOX) + 2 * k,
                    mndesc(ob + b * (BOX / 2), 1024) + 128 * k, id_z, (c | b | k) != 0);
            mma_commit(&S.o_empty[so]);
          }
          if (!ok) break;
          mma_commit(&S.a_empty[s]);
        }
        if (!ok) break;
        mma_commit(&S.z_full);
        for (int g = 0; ok && g < p.G; ++g, ++zu) {
          if (!wait_bar(&S.zp_full, zu & 1, abort_flag, 125)) { ok = false; break; }
          tc_fence_after();
          if (p.save_z) {
            tma_store(tm_zs[g], zp_tile, 0, tile * p.tt);
            bulk_commit();
          }
          for (int c = 0; c < p.nM[g]; ++c, ++io, ++yc) {
            const int so = io % QKV_NOP;
            const int yb = yc & 1;
            if (!wait_bar(&S.x_empty[yb], ((yc >> 1) & 1) ^ 1, abort_flag, 126)) { ok = false; break; }
            if (!wait_bar(&S.o_full[so], (io / QKV_NOP) & 1, abort_flag, 127)) { ok = false; break; }
            tc_fence_after();
            const uint32_t ob = su32(opr + so * BOX);
            for (int k = 0; k < p.kb[g]; ++k)
              mma(tmem + QF_Y + yb * 128, kdesc(zp_addr) + 2 * k, mndesc(ob, BOX / 2) + 128 * k,
                  id_y, k != 0);
            mma_commit(&S.o_empty[so]);
            mma_commit(&S.x_full[yb]);
          }
          if (!ok) break;
          if (p.save_z) bulk_wait_read<0>();
          mma_commit(&S.zp_empty);
        }
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
    uint8_t* my_stg = staging + (warp - 2) * 2 * STG;
    int yc = 0, tl = 0, zu = 0;
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++tl) {
      float v[32];
      bool ok = true;
      if (!warp_wait(&S.z_full, tl & 1, abort_flag, 128)) break;
      tc_fence_after();
      for (int g = 0; g < p.G; ++g, ++zu) {
        tmem_ld32(tmem + lane_off + QF_Z + 64 * g + 32 * h, v);
        if (g == p.G - 1) {  // every z_g is in registers or a tile by now
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.z_empty);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= S.Dc[g][32 * h + j];
        if (!warp_wait(&S.zp_empty, (zu & 1) ^ 1, abort_flag, 129)) { ok = false; break; }
        st_tile_half(zp_tile, row, h, v);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.zp_full);
        for (int c = 0; c < p.nM[g]; ++c, ++yc) {
          const int yb = yc & 1;
          if (!warp_wait(&S.x_full[yb], (yc >> 1) & 1, abort_flag, 130)) { ok = false; break; }
          tc_fence_after();
          uint8_t* box = my_stg + (yc & 1) * STG;
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
#pragma unroll
          for (int piece = 0; piece < 2; ++piece) {
            tmem_ld32(tmem + lane_off + QF_Y + yb * 128 + 64 * h + 32 * piece, v);
            stage_bf16_32(box, lane, piece, v);
          }
          tc_fence_before();
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&S.x_empty[yb]);
            const int col = c * CH + 64 * h;
            const int vq = p.tt - 32 * q;  // rows of this quadrant inside the tile
            if (col < p.M[g] && vq > 0 && (int64_t)tile * p.tt + 32 * q < p.T)
              tma_store(vq >= 32 ? tm_y[g] : tm_y16[g], box, col, tile * p.tt + 32 * q);
            bulk_commit();  // one group per chunk, empty if skipped
          }
        }
        if (!ok) break;
      }
      if (!ok) break;
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_free(tmem);
}


struct QkvBwdArgs {
  int64_t T;
  int G, nN, ntiles, N, tt;
  int nM[kMaxGroups];
  int M[kMaxGroups];
  int kb[kMaxGroups];
  const float* Dc[kMaxGroups];
  const int* rinfo[kMaxGroups];
  float* dDc[kMaxGroups];
  ZeroList zero;             // ranges set to 0 on the way (what the merges add into)
  // TT_DETERMINISTIC: every token sum goes to this CTA's own slot (rows
  // blockIdx.x * rows.. of each dA / dB map; dD into dDslot[g][CTA][quadrant]),
  // stored by the CTA's first tile and added to by its later ones in tile order
  int det;
  float* dDslot[kMaxGroups];
};

// TMEM columns of the backward
constexpr uint32_t QB_DZP = 0, QB_W = 64, QB_X = 256;  // W: two 64-column buffers; X: two 128

constexpr size_t kSmemQkvBwd = QKV_NACT * ACT_STAGE + QKV_NOP * BOX + kMaxGroups * BOX +
                               NEPI * STG + sizeof(QkvSmem) + 1024;
static_assert(kSmemQkvBwd <= 227 * 1024, "QKV backward smem");

__global__ void __launch_bounds__(NTHREADS, 1)
    qkv_bwd_kernel(const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_dy0,
                   const __grid_constant__ CUtensorMap tm_dy1,
                   const __grid_constant__ CUtensorMap tm_dy2,
                   const __grid_constant__ CUtensorMap tm_anr0,
                   const __grid_constant__ CUtensorMap tm_anr1,
                   const __grid_constant__ CUtensorMap tm_anr2,
                   const __grid_constant__ CUtensorMap tm_bm0,
                   const __grid_constant__ CUtensorMap tm_bm1,
                   const __grid_constant__ CUtensorMap tm_bm2,
                   const __grid_constant__ CUtensorMap tm_dx,
                   const __grid_constant__ CUtensorMap tm_dx16,
                   const __grid_constant__ CUtensorMap tm_dac0,
                   const __grid_constant__ CUtensorMap tm_dac1,
                   const __grid_constant__ CUtensorMap tm_dac2,
                   const __grid_constant__ CUtensorMap tm_dbc0,
                   const __grid_constant__ CUtensorMap tm_dbc1,
                   const __grid_constant__ CUtensorMap tm_dbc2,
                   const __grid_constant__ CUtensorMap tm_zs0,
                   const __grid_constant__ CUtensorMap tm_zs1,
                   const __grid_constant__ CUtensorMap tm_zs2, QkvBwdArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1k(smem_raw);
  uint8_t* act = base;
  uint8_t* opr = act + QKV_NACT * ACT_STAGE;
  uint8_t* ztiles = opr + QKV_NOP * BOX;            // z'_g, then dz_g, one tile a layer
  uint8_t* staging = ztiles + kMaxGroups * BOX;     // one box per epilogue warp
  QkvSmem& S = *reinterpret_cast<QkvSmem*>(staging + NEPI * STG);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const CUtensorMap* tm_dy[kMaxGroups] = {&tm_dy0, &tm_dy1, &tm_dy2};
  const CUtensorMap* tm_anr[kMaxGroups] = {&tm_anr0, &tm_anr1, &tm_anr2};
  const CUtensorMap* tm_bm[kMaxGroups] = {&tm_bm0, &tm_bm1, &tm_bm2};
  const CUtensorMap* tm_dac[kMaxGroups] = {&tm_dac0, &tm_dac1, &tm_dac2};
  const CUtensorMap* tm_dbc[kMaxGroups] = {&tm_dbc0, &tm_dbc1, &tm_dbc2};
  const CUtensorMap* tm_zs[kMaxGroups] = {&tm_zs0, &tm_zs1, &tm_zs2};

  if (threadIdx.x == 0) {
    for (int s = 0; s < QKV_NACT; ++s) {
      mbar_init(&S.a_full[s], 1);
      mbar_init(&S.a_empty[s], 1);
    }
    for (int s = 0; s < QKV_NOP; ++s) {
      mbar_init(&S.o_full[s], 1);
      mbar_init(&S.o_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.x_full[b], 1);
      mbar_init(&S.x_empty[b], NEPI);
      mbar_init(&S.w_full[b], 1);
      mbar_init(&S.w_empty[b], NEPI);
    }
    mbar_init(&S.zl_full, 1);
    mbar_init(&S.zt_empty, 1);
    mbar_init(&S.dzp_full, 1);
    mbar_init(&S.dzp_empty, NEPI);
    mbar_init(&S.dz_full, NEPI);
    mbar_init(&S.fin, 1);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(&S.tmem_base);
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < p.G * RP; i += blockDim.x) S.Dc[i / RP][i % RP] = p.Dc[i / RP][i % RP];
  zero_list(p.zero);
  zero_tail_boxes(act, 2 * QKV_NACT, ztiles, kMaxGroups, p.tt);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort_flag = &S.abort_flag;

  if (warp == 0) {
    // ---------------- TMA producer: the z'_g tiles, each layer's dy chunks
    // (with its B columns), then the x chunks (with every layer's A rows)
    if (lane == 0) {
      int ia = 0, io = 0, tl = 0;
      int lpa[QKV_NACT], lpo[QKV_NOP];
      for (int s = 0; s < QKV_NACT; ++s) lpa[s] = -1;
      for (int s = 0; s < QKV_NOP; ++s) lpo[s] = -1;
      bool ok = true;
      auto take_act = [&](int& s) -> bool {
        s = ia % QKV_NACT;
        const uint32_t ph = (ia / QKV_NACT) & 1;
        if (!wait_bar(&S.a_empty[s], ph ^ 1, abort_flag, 140)) return false;
        lpa[s] = (int)ph;
        ++ia;
        return true;
      };
      auto take_op = [&](int& s) -> bool {
        s = io % QKV_NOP;
        const uint32_t ph = (io / QKV_NOP) & 1;
        if (!wait_bar(&S.o_empty[s], ph ^ 1, abort_flag, 141)) return false;
        lpo[s] = (int)ph;
        ++io;
        return true;
      };
      const uint32_t act_bytes = (uint32_t)p.tt * 128;  // one activation box of tt rows
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x, ++tl) {
        const int tok0 = tile * p.tt;
        if (!wait_bar(&S.zt_empty, (tl & 1) ^ 1, abort_flag, 142)) break;
        mbar_expect_tx(&S.zl_full, p.G * act_bytes);
        for (int g = 0; g < p.G; ++g) tma_load(ztiles + g * BOX, tm_zs[g], &S.zl_full, 0, tok0);
        for (int g = 0; ok && g < p.G; ++g)
          for (int c = 0; c < p.nM[g]; ++c) {
            const int col = rot_chunk(c, p.nM[g], tile) * CH;
            int sa, so;
            if (!take_act(sa)) { ok = false; break; }
            mbar_expect_tx(&S.a_full[sa], 2 * act_bytes);
            tma_load(act + sa * ACT_STAGE, tm_dy[g], &S.a_full[sa], col, tok0);
            tma_load(act + sa * ACT_STAGE + BOX, tm_dy[g], &S.a_full[sa], col + 64, tok0);
            if (!take_op(so)) { ok = false; break; }
            mbar_expect_tx(&S.o_full[so], BOX);
            tma_load(opr + so * BOX, tm_bm[g], &S.o_full[so], col, 0);
            tma_load(opr + so * BOX + BOX / 2, tm_bm[g], &S.o_full[so], col + 64, 0);
          }
        for (int c = 0; ok && c < p.nN; ++c) {
          const int col = rot_chunk(c, p.nN, tile) * CH;
          int sa;
          if (!take_act(sa)) { ok = false; break; }
          mbar_expect_tx(&S.a_full[sa], 2 * act_bytes);
          tma_load(act + sa * ACT_STAGE, &tm_x, &S.a_full[sa], col, tok0);
          tma_load(act + sa * ACT_STAGE + BOX, &tm_x, &S.a_full[sa], col + 64, tok0);
          for (int g = 0; g < p.G; ++g) {
            int so;
            if (!take_op(so)) { ok = false; break; }
            mbar_expect_tx(&S.o_full[so], BOX);
            tma_load(opr + so * BOX, tm_anr[g], &S.o_full[so], 0, col);
          }
        }
      }
      for (int s = 0; s < QKV_NACT; ++s)
        if (lpa[s] >= 0) drain_bar(&S.a_full[s], (uint32_t)lpa[s]);
      for (int s = 0; s < QKV_NOP; ++s)
        if (lpo[s] >= 0) drain_bar(&S.o_full[s], (uint32_t)lpo[s]);
      if (tl > 0) drain_bar(&S.zl_full, (uint32_t)((tl - 1) & 1));
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_r = idesc(128, 64, 0, 0);    // token x rank, K-major
      const uint32_t id_w = idesc(128, 64, 1, 1);    // weight x rank, MN-major
      const uint32_t id_x = idesc(128, 128, 0, 0);   // token x feature, K = rank
      const uint32_t zt = su32(ztiles);
      int ia = 0, io = 0, wc = 0, xc = 0, tl = 0, dzu = 0;
      bool ok = true;
      auto w_take = [&](uint32_t& col) -> bool {
        const int wb = wc & 1;
        if (!wait_bar(&S.w_empty[wb], ((wc >> 1) & 1) ^ 1, abort_flag, 143)) return false;
        tc_fence_after();
        col = tmem + QB_W + wb * 64;
        return true;
      };
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x, ++tl) {
        if (!wait_bar(&S.zl_full, tl & 1, abort_flag, 144)) break;
        // B (each layer): dz'_g = dy_g B_g^T ; dB_g^T chunk = dy_g^T z'_g
        for (int g = 0; ok && g < p.G; ++g, ++dzu) {
          if (!wait_bar(&S.dzp_empty, (dzu & 1) ^ 1, abort_flag, 145)) { ok = false; break; }
          tc_fence_after();
          const uint32_t zg = zt + g * BOX;
          for (int c = 0; c < p.nM[g]; ++c, ++ia, ++io) {
            const int sa = ia % QKV_NACT, so = io % QKV_NOP;
            if (!wait_bar(&S.a_full[sa], (ia / QKV_NACT) & 1, abort_flag, 146)) { ok = false; break; }
            if (!wait_bar(&S.o_full[so], (io / QKV_NOP) & 1, abort_flag, 147)) { ok = false; break; }
            tc_fence_after();
            const uint32_t st = su32(act + sa * ACT_STAGE), ob = su32(opr + so * BOX);
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma(tmem + QB_DZP, kdesc(st + b * BOX) + 2 * k, kdesc(ob + b * (BOX / 2)) + 2 * k,
                    id_r, (c | b | k) != 0);
            uint32_t wcol;
            if (!w_take(wcol)) { ok = false; break; }
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma(wcol, mndesc(st, BOX) + 128 * k, mndesc(zg, 1024) + 128 * k, id_w, k != 0);
            mma_commit(&S.w_full[wc & 1]);
            ++wc;
            mma_commit(&S.o_empty[so]);
            mma_commit(&S.a_empty[sa]);
          }
          if (!ok) break;
          mma_commit(&S.dzp_full);  // also: this layer's z'_g readers are done
        }
        if (!ok) break;
        // C: dx = sum_g dz_g A_g^T ; dA_g chunk = x^T dz_g
        if (!wait_bar(&S.dz_full, tl & 1, abort_flag, 148)) break;
        tc_fence_after();
        for (int c = 0; c < p.nN; ++c, ++ia, ++xc) {
          const int sa = ia % QKV_NACT;
          const int xb = xc & 1;
          if (!wait_bar(&S.a_full[sa], (ia / QKV_NACT) & 1, abort_flag, 149)) { ok = false; break; }
          if (!wait_bar(&S.x_empty[xb], ((xc >> 1) & 1) ^ 1, abort_flag, 150)) { ok = false; break; }
          const uint32_t st = su32(act + sa * ACT_STAGE);
          // every layer's dx term first, so that the dx chunk is handed over
          // before the W buffers (the epilogue drains in this order)
          for (int g = 0; g < p.G; ++g, ++io) {
            const int so = io % QKV_NOP;
            if (!wait_bar(&S.o_full[so], (io / QKV_NOP) & 1, abort_flag, 151)) { ok = false; break; }
            tc_fence_after();
            const uint32_t ob = su32(opr + so * BOX);
            for (int k = 0; k < p.kb[g]; ++k)
              mma(tmem + QB_X + xb * 128, kdesc(zt + g * BOX) + 2 * k, kdesc(ob) + 2 * k, id_x,
                  (g | k) != 0);
            mma_commit(&S.o_empty[so]);
          }
          if (!ok) break;
          mma_commit(&S.x_full[xb]);
          for (int g = 0; g < p.G; ++g) {
            uint32_t wcol;
            if (!w_take(wcol)) { ok = false; break; }
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma(wcol, mndesc(st, BOX) + 128 * k, mndesc(zt + g * BOX, 1024) + 128 * k, id_w,
                  k != 0);
            mma_commit(&S.w_full[wc & 1]);
            ++wc;
          }
          if (!ok) break;
          mma_commit(&S.a_empty[sa]);
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
    uint8_t* box = staging + (warp - 2) * STG;
    int rp[kMaxGroups];
    for (int g = 0; g < kMaxGroups; ++g) rp[g] = g < p.G ? p.rinfo[g][0] : 0;
    int wc = 0, xc = 0, tl = 0, dzu = 0;
    // the next W buffer: rows row0 + 32 q, rank columns 32 h, bulk-added into map
    auto drain_w = [&](const CUtensorMap* map, int row0, int nrows, int rprime) -> bool {
      float v[32];
      const int wb = wc & 1;
      if (!warp_wait(&S.w_full[wb], (wc >> 1) & 1, abort_flag, 152)) return false;
      tc_fence_after();
      tmem_ld32(tmem + lane_off + QB_W + wb * 64 + 32 * h, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.w_empty[wb]);
      ++wc;
      if (32 * h < rprime && row0 + 32 * q < nrows) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        stage_f32_32(box, lane, v);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int r = (p.det ? (int)blockIdx.x * nrows : 0) + row0 + 32 * q;
          if (p.det && tl == 0)
            tma_store(map, box, 32 * h, r);
          else
            tma_reduce_add(map, box, 32 * h, r);
          bulk_commit();
        }
      }
      return true;
    };
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++tl) {
      bool ok = true;
      for (int g = 0; ok && g < p.G; ++g, ++dzu) {
        float z[32], v[32];
        for (int c = 0; c < p.nM[g]; ++c)
          if (!drain_w(tm_dbc[g], rot_chunk(c, p.nM[g], tile) * CH, p.M[g], rp[g])) {
            ok = false;
            break;
          }
        if (!ok) break;
        // dz'_g -> dD_g, dz_g tile (over z'_g, whose readers are done)
        if (!warp_wait(&S.dzp_full, dzu & 1, abort_flag, 153)) { ok = false; break; }
        tc_fence_after();
        tmem_ld32(tmem + lane_off + QB_DZP + 32 * h, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.dzp_empty);
        if (!warp_wait(&S.zl_full, tl & 1, abort_flag, 154)) { ok = false; break; }
        uint8_t* ztile = ztiles + g * BOX;
        ld_tile_half(ztile, row, h, z);
        {
          float pr[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) pr[j] = z[j] * v[j];
          const float colsum = warp_transpose_sum(pr, lane);
          if (32 * h + lane < rp[g]) {
            const float d = colsum / S.Dc[g][32 * h + lane];
            if (p.det) {  // this lane alone owns the entry of its CTA and quadrant
              float* e = p.dDslot[g] + ((size_t)blockIdx.x * 4 + q) * RP + 32 * h + lane;
              *e = tl == 0 ? d : *e + d;
            } else {
              atomicAdd(p.dDc[g] + 32 * h + lane, d);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= S.Dc[g][32 * h + j];
        __syncwarp();
        st_tile_half(ztile, row, h, v);
        fence_async_smem();
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mbar_arrive(&S.dz_full);
      // dx chunks and every layer's dA chunks
      for (int c = 0; c < p.nN; ++c, ++xc) {
        float v[32];
        const int xb = xc & 1;
        if (!warp_wait(&S.x_full[xb], (xc >> 1) & 1, abort_flag, 155)) { ok = false; break; }
        tc_fence_after();
        const int cx = rot_chunk(c, p.nN, tile);
        const int col = cx * CH + 64 * h;
        const int vq = p.tt - 32 * q;  // rows of this quadrant inside the tile
        const bool st_dx = col < p.N && vq > 0 && (int64_t)tile * p.tt + 32 * q < p.T;
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {
          tmem_ld32(tmem + lane_off + QB_X + xb * 128 + 64 * h + 32 * piece, v);
          stage_bf16_32(box, lane, piece, v);
        }
        tc_fence_before();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&S.x_empty[xb]);
          if (st_dx) {
            tma_store(vq >= 32 ? &tm_dx : &tm_dx16, box, col, tile * p.tt + 32 * q);
            bulk_commit();
          }
        }
        for (int g = 0; g < p.G; ++g)
          if (!drain_w(tm_dac[g], cx * CH, p.N, rp[g])) { ok = false; break; }
        if (!ok) break;
      }
      if (!ok) break;
      // the next tile's adds into this CTA's slots come after this tile's
      if (p.det && lane == 0) bulk_wait_all();
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_free(tmem);
}

// 16-rank blocks of the padded middle rank that can hold a nonzero column
// (the columns past r_d are zero in z', dz and the packed operands)
int kblocks(const LayerPlan& L) {
  const int r = L.rd < RP ? L.rd : RP;
  return r > 0 ? (r + 15) >> 4 : 1;
}

cudaError_t set_qkv_attrs() {
  static PerDevice once;
  return once.get([] {
    cudaError_t e = cudaFuncSetAttribute(qkv_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemQkvFwd);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(qkv_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemQkvBwd);
    return e;
  });
}

}  // namespace

bool multi_tc_supported(const LayerPlan* Ls, int G) {
  if (G < 1 || G > kMaxGroups) return false;
  for (int g = 0; g < G; ++g)
    if (!tc_supported(Ls[g]) || Ls[g].N != Ls[0].N) return false;
  return true;
}

tt_status multi_tc_forward(const LayerPlan* Ls, int G, int64_t T, const void* x, void* const* y,
                           void* ws, const size_t* offs, void* const* zs, bool prefetch_x,
                           cudaStream_t st) {
  if (T <= 0) return TT_OK;
  if (T > (int64_t)0x7FFFFFFF - TILE || !multi_tc_supported(Ls, G)) return TT_ERR_UNSUPPORTED;
  if (set_qkv_attrs() != cudaSuccess) return TT_ERR_CUDA;
  const bool keep = zs != nullptr;
  CUtensorMap mx, manr[kMaxGroups], mbm[kMaxGroups], my[kMaxGroups], my16[kMaxGroups],
      mzs[kMaxGroups];
  QkvFwdArgs a;
  a.T = T;
  a.G = G;
  a.nN = (int)((Ls[0].N + CH - 1) / CH);
  a.tt = tokens_per_tile(T);
  a.ntiles = (int)((T + a.tt - 1) / a.tt);
  a.save_z = keep ? 1 : 0;
  a.prefetch_x = prefetch_x && pdl_enabled() ? 1 : 0;
  if (!make_map(&mx, x, Ls[0].N, T, 64, a.tt)) return TT_ERR_CUDA;
  for (int g = 0; g < kMaxGroups; ++g) {
    const int gg = g < G ? g : 0;  // unused slots repeat layer 0's maps
    const LayerPlan& L = Ls[gg];
    const TcLayout t = tc_layout(L);
    void* yy = y ? y[gg] : nullptr;
    void* zz = keep ? zs[gg] : nullptr;
    void* any = yy ? yy : zz;
    if (!any) return TT_ERR_INVALID_ARG;
    if (!make_map(&manr[g], at<void>(ws, offs[gg] + t.Anr), RP, L.N, 64, CH) ||
        !make_map(&mbm[g], at<void>(ws, offs[gg] + t.Bm), L.M, RP, 64, RP) ||
        !make_map(&my[g], yy ? yy : any, yy ? L.M : RP, T, 64, 32) ||
        !make_map(&my16[g], yy ? yy : any, yy ? L.M : RP, T, 64, 16) ||
        !make_map(&mzs[g], zz ? zz : any, RP, T, 64, a.tt))
      return TT_ERR_CUDA;
    a.nM[g] = (y && g < G) ? (int)((L.M + CH - 1) / CH) : 0;  // no y: the kept z' only
    a.M[g] = (int)L.M;
    a.kb[g] = kblocks(L);
    a.Dc[g] = at<float>(ws, offs[gg] + t.Dc);
  }
  const int grid = a.ntiles < num_sms() ? a.ntiles : num_sms();
  cudaError_t e = launch_ex(qkv_fwd_kernel, grid, NTHREADS, kSmemQkvFwd, st, false, mx, manr[0],
                            manr[1], manr[2], mbm[0], mbm[1], mbm[2], my[0], my[1], my[2], my16[0],
                            my16[1], my16[2], mzs[0], mzs[1], mzs[2], a);
  count_launches(1);
  return e == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

tt_status multi_tc_backward(const LayerPlan* Ls, int G, int64_t T, const void* x,
                            const void* const* dy, void* dx, void* ws, const size_t* offs,
                            const void* const* zs, const ZeroList& zero, const DetSlots* det,
                            cudaStream_t st) {
  if (!multi_tc_supported(Ls, G)) return TT_ERR_UNSUPPORTED;
  if (T <= 0) return zero_list_memset(zero, st) == cudaSuccess ? TT_OK : TT_ERR_CUDA;
  if (T > (int64_t)0x7FFFFFFF - TILE) return TT_ERR_UNSUPPORTED;
  if (det)
    for (int g = 0; g < G; ++g)
      if (det[g].count < 1 || det[g].count != det[0].count ||
          (int64_t)det[g].count * (Ls[g].N > Ls[g].M ? Ls[g].N : Ls[g].M) > 0x7FFFFFFF)
        return TT_ERR_UNSUPPORTED;
  const int64_t nslot = det ? det[0].count : 1;
  if (set_qkv_attrs() != cudaSuccess) return TT_ERR_CUDA;
  CUtensorMap mx, mdx, mdx16, mdy[kMaxGroups], manr[kMaxGroups], mbm[kMaxGroups], mdac[kMaxGroups],
      mdbc[kMaxGroups], mzs[kMaxGroups];
  QkvBwdArgs a;
  a.T = T;
  a.G = G;
  a.N = (int)Ls[0].N;
  a.nN = (int)((Ls[0].N + CH - 1) / CH);
  // a fixed summation order wants a fixed token blocking: 128-token tiles
  a.tt = det ? TILE : tokens_per_tile(T);
  a.ntiles = (int)((T + a.tt - 1) / a.tt);
  if (!make_map(&mx, x, Ls[0].N, T, 64, a.tt) || !make_map(&mdx, dx, Ls[0].N, T, 64, 32) ||
      !make_map(&mdx16, dx, Ls[0].N, T, 64, 16))
    return TT_ERR_CUDA;
  for (int g = 0; g < kMaxGroups; ++g) {
    const int gg = g < G ? g : 0;
    const LayerPlan& L = Ls[gg];
    const TcLayout t = tc_layout(L);
    if (!make_map(&mdy[g], dy[gg], L.M, T, 64, a.tt) ||
        !make_map(&manr[g], at<void>(ws, offs[gg] + t.Anr), RP, L.N, 64, CH) ||
        !make_map(&mbm[g], at<void>(ws, offs[gg] + t.Bm), L.M, RP, 64, RP) ||
        !make_map(&mdac[g], det ? det[gg].a : at<void>(ws, offs[gg] + t.dAc), RP, L.N * nslot,
                  32, 32, kMapF32) ||
        !make_map(&mdbc[g], det ? det[gg].b : at<void>(ws, offs[gg] + t.dBc), RP, L.M * nslot,
                  32, 32, kMapF32) ||
        !make_map(&mzs[g], zs[gg], RP, T, 64, a.tt))
      return TT_ERR_CUDA;
    a.nM[g] = (int)((L.M + CH - 1) / CH);
    a.M[g] = (int)L.M;
    a.kb[g] = kblocks(L);
    a.Dc[g] = at<float>(ws, offs[gg] + t.Dc);
    a.rinfo[g] = at<int>(ws, offs[gg] + t.rinfo);
    a.dDc[g] = at<float>(ws, offs[gg] + t.dDc);
    a.dDslot[g] = det ? det[gg].d : nullptr;
  }
  a.zero = zero;
  a.det = det ? 1 : 0;
  int grid = a.ntiles < num_sms() ? a.ntiles : num_sms();
  if (det && grid > det[0].count) grid = det[0].count;
  cudaError_t e = launch_ex(qkv_bwd_kernel, grid, NTHREADS, kSmemQkvBwd, st, false, mx, mdy[0],
                            mdy[1], mdy[2], manr[0], manr[1], manr[2], mbm[0], mbm[1], mbm[2],
                            mdx, mdx16, mdac[0], mdac[1], mdac[2], mdbc[0], mdbc[1], mdbc[2], mzs[0],
                            mzs[1], mzs[2], a);
  count_launches(1);
  if (e != cudaSuccess) return TT_ERR_CUDA;
  if (det)  // each layer's slots of the `grid` CTAs, summed in CTA order
    for (int g = 0; g < G && e == cudaSuccess; ++g) {
      const TcLayout t = tc_layout(Ls[g]);
      e = det_sum_launch(Ls[g], det[g], grid, at<float>(ws, offs[g] + t.dAc),
                         at<float>(ws, offs[g] + t.dBc), a.dDc[g], st);
    }
  return e == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

}  // namespace ttc
