// Fused token-tile kernels for bf16 activations on sm_103a: tcgen05 MMAs with
// TMEM accumulators, TMA (128-byte swizzle) staging, mbarrier pipelines.
//
// The contraction order is the one of the CoMERA project page ("Making small
// tensor operations fast on GPUs", bullet "One contraction order for both
// passes"): the merged input side A (N x r) and output side B (r x M) are
// applied to a tile of 128 tokens at a time, and the rank-r intermediates
// z = x A, z' = z diag(D_d), dz' = dy B^T, dz = dz' diag(D_d) never leave the
// SM (TMEM and shared memory).
//
// Layout of the packed operands (bf16, rank padded to RP = 64 with zero rows
// or columns; the middle rank is compacted to the nonzero entries of D_d, so
// pruned ranks cost nothing but padding):
//   Anr (N x RP)  B operand of z  = x  . A     (K = features, MN-major)
//                 and of dx = dz . Anr^T      (K = rank, K-major)
//   Bm  (RP x M)  B operand of y  = z' . Bm    (K = rank, MN-major)
//                 and of dz'= dy . Bm^T       (K = outputs, K-major)
// Each is stored once, in the layout whose rows the merges write contiguously;
// a 128-byte swizzled box of it serves as either operand major-ness.  The
// weight-side products dA = x^T dz and dB^T = dy^T z' read the very same
// x / dy / z' / dz tiles through MN-major descriptors (the 128-byte swizzled
// [token][64 elements] tile is K-major for the token-side products and
// MN-major for the weight-side ones).
//
// FP8 activations: with E4M3 x and dy (one byte an element) the same kernels
// run with four more warps.  TMA brings each 128-token x 128-column E4M3 tile
// into the second half of a stage's activation area; the converter warps
// widen it in place to the two bf16 boxes the MMAs read (E4M3 values are
// exact in bf16), so the tensor-core work and everything downstream is the
// bf16 path's, and only the activation bytes read from HBM halve.
//
// Every mbarrier wait is bounded (global timer); on expiry the CTA records
// TT_ERR_TIMEOUT in the per-device status word, raises a shared abort flag so
// the other roles stop, waits (bounded) for its own copies and MMAs, frees its
// TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdlib>
#include <mutex>
#include <utility>

#include "tc_fused.h"

namespace ttc {

__device__ DeviceStatus g_status;
// Limit of every bounded device wait (ns on the global timer), and the test
// hook that makes one arrival go missing (tt_set_wait_limit_ns,
// tt_debug_skip_arrival).
__device__ unsigned long long g_wait_limit_ns = 2000000000ull;
__device__ int g_debug_skip = 0;

cudaError_t read_and_clear_device_status(DeviceStatus* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(DeviceStatus));
  if (e != cudaSuccess) return e;
  DeviceStatus z{0, 0};
  return cudaMemcpyToSymbol(g_status, &z, sizeof(z));
}

namespace {

constexpr int TILE = 128;            // MMA M: rows of a token tile in shared memory and TMEM
constexpr int RP = 64;               // padded rank (one 128-byte swizzle atom)
constexpr int CH = 128;              // features / outputs per pipeline chunk
constexpr int BOX = 16 * 1024;       // [128 rows][64 bf16] swizzled box
constexpr int STAGE = 48 * 1024;     // 2 activation boxes + 16 KB operand
constexpr int OPND = 32 * 1024;      // operand offset inside a stage
constexpr int NSTAGE_F = 3;
constexpr int NSTAGE_B = 3;
constexpr int NEPI = 8;              // epilogue warps
constexpr int STG = 4096;            // one epilogue staging box: 32 rows x 128 bytes
constexpr int NTHREADS = (2 + NEPI) * 32;
constexpr int NCONV = 4;             // E4M3 -> bf16 converter warps (FP8 kernels)
constexpr int NTHREADS_F8 = (2 + NEPI + NCONV) * 32;

// TMEM columns
constexpr uint32_t F_Z = 0, F_Y = 128;                       // forward
constexpr uint32_t B_Z = 0, B_DZP = 64, B_W = 128, B_X = 256;  // backward
constexpr uint32_t TMEM_COLS = 512;

// --------------------------------------------------------------------------
// PTX helpers

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Optional per-CTA timeline (global-timer stamps), compiled in only with
// -DTTC_TIMELINE for performance investigation; the default build has none.
#ifdef TTC_TIMELINE
__device__ unsigned long long g_tl[4][256][16];  // fwd, bwd, engine (1 phase), engine (more)
__device__ unsigned long long g_tlu[256][8][8];  // engine units: (phase*100+task, start, end, inner stamps)
#define TL_STAMP(k, slot) (g_tl[(k)][blockIdx.x & 255][(slot)] = gtimer())
// per-warp stamps of the backward token kernel's CTA 0: [warp][slot]
__device__ unsigned long long g_tlk[16][48];
#define TLK(slot) \
  if (blockIdx.x == 0 && (threadIdx.x & 31) == 0 && (slot) < 48) g_tlk[threadIdx.x >> 5][(slot)] = gtimer()
#define TLU_STAMP(nu, slot) \
  if (threadIdx.x == 0 && (nu) < 8) g_tlu[blockIdx.x & 255][(nu)][(slot)] = gtimer()
#else
#define TLU_STAMP(nu, slot) ((void)0)
#define TL_STAMP(k, slot) ((void)0)
#define TLK(slot) ((void)0)
#endif

__device__ void record_error(unsigned code, unsigned where) {
  if (atomicCAS(&g_status.code, 0u, code) == 0u) atomicExch(&g_status.detail, where);
}

// True (once) when the test hook asks this launch to skip one arrival.
__device__ __forceinline__ bool debug_take(int site) {
  return *(volatile int*)&g_debug_skip == site && atomicCAS(&g_debug_skip, site, 0) == site;
}

// Wait for the phase of the given parity; false if aborted or timed out.
__device__ __forceinline__ bool wait_bar(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                         unsigned where) {
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = gtimer();
  const uint64_t limit = *(volatile unsigned long long*)&g_wait_limit_ns;
  while (!mbar_try_wait(b, parity)) {
    if (*abort_flag) return false;
    if (gtimer() - t0 > limit) {
      *abort_flag = 1;
      record_error(TT_ERR_TIMEOUT, where);
      return false;
    }
  }
  return true;
}

// Warp-uniform wait: lane 0 polls, the result is broadcast, so that the
// warp stays converged for the .sync.aligned TMEM loads that follow.
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                          unsigned where) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(b, parity, abort_flag, where) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Drain wait used on the way out: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_bar(uint64_t* b, uint32_t parity) {
  const uint64_t t0 = gtimer();
  const uint64_t limit = *(volatile unsigned long long*)&g_wait_limit_ns / 4;
  while (!mbar_try_wait(b, parity)) {
    if (gtimer() - t0 > limit) return;
  }
}

__device__ __forceinline__ void tma_load(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                         int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(su32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// Programmatic dependent launch: wait for the grids this one depends on
// (their memory is visible afterwards), and let the next grid in the stream
// be scheduled early.  Both are no-ops for a grid launched without the
// programmatic-serialization attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// smem matrix descriptor, 128-byte swizzle, sm_100 family (version 1)
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ uint64_t kdesc(uint32_t saddr) { return sdesc(saddr, 16, 1024); }
__device__ __forceinline__ uint64_t mndesc(uint32_t saddr, uint32_t lbo) {
  return sdesc(saddr, lbo, 1024);
}

// instruction descriptor: bf16 x bf16 -> f32, dense
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t id,
                                    uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(dtmem),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          su32(bar))
      : "memory");
}

#define TT_LD32_REGS                                                                         \
  "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, " \
  "%19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}"

// 32 consecutive f32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " TT_LD32_REGS ", [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                 "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                 "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                 "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                 "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Write 32 values (columns [32h, 32h+32) of row `row`) as bf16 into a
// [128][64] tile in the 128-byte swizzled layout used by TMA and the MMAs.
__device__ __forceinline__ void st_tile_half(uint8_t* tile, int row, int h, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
    u.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
    u.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
    u.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
    const int chunk = (4 * h + q) ^ (row & 7);
    *reinterpret_cast<uint4*>(tile + row * 128 + chunk * 16) = u;
  }
}

// Inverse of st_tile_half: columns [32h, 32h+32) of row `row` as f32.
__device__ __forceinline__ void ld_tile_half(const uint8_t* tile, int row, int h, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int chunk = (4 * h + q) ^ (row & 7);
    const uint4 u = *reinterpret_cast<const uint4*>(tile + row * 128 + chunk * 16);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      v[8 * q + 2 * i] = f.x;
      v[8 * q + 2 * i + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void tma_store(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(su32(src)), "r"(c0), "r"(c1)
      : "memory");
}

// Element-wise atomic add of a shared-memory box into global memory.
__device__ __forceinline__ void tma_reduce_add(const CUtensorMap* map, const void* src, int c0,
                                               int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(su32(src)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups of this thread still read smem.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Staging boxes are [32 rows][128 bytes] with the 128-byte swizzle the
// tensor maps use: 16-byte chunk q of row r lives at r*128 + (q ^ (r & 7))*16.
__device__ __forceinline__ void stage_bf16_32(uint8_t* box, int r, int piece,
                                              const float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 u;
    u.x = pack_bf16(v[8 * i + 0], v[8 * i + 1]);
    u.y = pack_bf16(v[8 * i + 2], v[8 * i + 3]);
    u.z = pack_bf16(v[8 * i + 4], v[8 * i + 5]);
    u.w = pack_bf16(v[8 * i + 6], v[8 * i + 7]);
    const int q = 4 * piece + i;
    *reinterpret_cast<uint4*>(box + r * 128 + ((q ^ (r & 7)) << 4)) = u;
  }
}
__device__ __forceinline__ void stage_f32_32(uint8_t* box, int r, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 f = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    *reinterpret_cast<float4*>(box + r * 128 + ((q ^ (r & 7)) << 4)) = f;
  }
}

// After the butterfly, lane l holds sum over the warp's 32 lanes of v[l].
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

// Two E4M3 codes (low byte first) -> two bf16 values (low half first).
// Every E4M3 value is exact in f16, f32 and bf16, so no rounding happens.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  return pack_bf16(f.x, f.y);
}

// Widen the 128-row x 128-column E4M3 tile that TMA wrote (128-byte swizzle)
// at st + BOX into the two [128][64] bf16 boxes at st and st + BOX.  Converter
// warp cw owns rows 32cw .. 32cw + 31: the bf16 rows it writes into the second
// box occupy exactly the bytes of the raw rows it read, so the warp reads all
// of its raw bytes into registers, syncs, and only then writes.
__device__ __forceinline__ void widen_e4m3_tile(uint8_t* st, int cw, int lane) {
  const uint8_t* raw = st + BOX + cw * 32 * 128;
  uint4 u[8];
#pragma unroll
  for (int n = 0; n < 8; ++n)
    u[n] = *reinterpret_cast<const uint4*>(raw + (n * 32 + lane) * 16);
  __syncwarp();
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const int unit = n * 32 + lane;      // physical 16-byte unit of the warp's rows
    const int r = cw * 32 + (unit >> 3);
    const int j = (unit & 7) ^ (r & 7);  // columns 16j .. 16j + 15
    uint8_t* dst = st + (j >> 2) * BOX + r * 128;
    const int k0 = 2 * (j & 3);          // their first bf16 16-byte chunk in that box
    uint4 o0, o1;
    o0.x = e4m3x2_to_bf16x2(u[n].x);
    o0.y = e4m3x2_to_bf16x2(u[n].x >> 16);
    o0.z = e4m3x2_to_bf16x2(u[n].y);
    o0.w = e4m3x2_to_bf16x2(u[n].y >> 16);
    o1.x = e4m3x2_to_bf16x2(u[n].z);
    o1.y = e4m3x2_to_bf16x2(u[n].z >> 16);
    o1.z = e4m3x2_to_bf16x2(u[n].w);
    o1.w = e4m3x2_to_bf16x2(u[n].w >> 16);
    *reinterpret_cast<uint4*>(dst + ((k0 ^ (r & 7)) << 4)) = o0;
    *reinterpret_cast<uint4*>(dst + (((k0 + 1) ^ (r & 7)) << 4)) = o1;
  }
}

// A tile holds tt <= TILE tokens (a multiple of 16, chosen on the host so that
// the tiles spread over every SM); rows tt .. TILE-1 of the shared-memory
// activation boxes are zeroed once and never written by TMA, so they add
// nothing to the token sums.
struct FwdArgs {
  int64_t T;
  int N, M, nN, nM, ntiles, tt;
  int save_z;  // also store each tile's z' (bf16 [T][64]) through tm_zs
  // the grid before this one is the merge of the same call, which does not
  // write x: the first stages' x boxes are requested before the dependency wait
  int prefetch_x;
  const float* Dc;
  __nv_bfloat16* y;
};

struct BwdArgs {
  int64_t T;
  int N, M, nN, nM, ntiles, tt;
  const float* Dc;
  const int* rinfo;  // [0] = r', [1..64] = kept index of each compacted column
  __nv_bfloat16* dx;
  float* dAc;  // N x RP
  float* dBc;  // M x RP
  float* dDc;  // RP
  ZeroList zero;  // ranges set to 0 on the way (what the merge backward adds into)
  int use_z;    // read the forward's z' through tm_zs instead of computing x A
  // Fixed summation order: the token sums go to this CTA's own slot (rows
  // blockIdx.x * N of tm_dac, blockIdx.x * M of tm_dbc; dDslot[blockIdx.x][4
  // quadrants][64]), stored by the CTA's first tile and added to by its later
  // ones, each tile's bulk operations completed before the next tile's.
  int det;
  float* dDslot;
};

struct SmemCommon {
  uint64_t full[4], empty[4];
  uint64_t z_full, z_empty, zp_full, zp_empty, dzp_full, dzp_empty, dz_full, dz_empty;
  uint64_t w_full[2], w_empty[2], x_full[2], x_empty[2];
  uint64_t conv[4];  // FP8 kernels: stage s converted (and its operand loaded)
  uint64_t zl_full;  // backward with a kept z': the z' tile has landed
  uint64_t fin;
  uint32_t tmem_base;
  int abort_flag;
  float Dc[RP];
};

// Chunk i of n visited in position c of a tile's phase.  The backward's
// token sums are bulk-added into one [N or M][64] buffer by every CTA; with
// the order rotated by the tile index, concurrent CTAs add into different
// row blocks instead of all into the same one.
__device__ __forceinline__ int rot_chunk(int c, int n, int tile) {
  const int i = c + tile % n;
  return i < n ? i : i - n;
}

// Zero rows [tt, TILE) of the stages' two activation boxes and of the z' tile.
// Every range of the list set to 0, grid-stride over the whole grid.
__device__ void zero_list(const ZeroList& z) {
  const int stride = gridDim.x * blockDim.x;
  for (int r = 0; r < z.count; ++r)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < z.n[r]; i += stride) z.p[r][i] = 0.f;
}

// The compacted middle rank r' (the nonzero entries of Dc come first) and the
// 16-wide K blocks of the rank dimension that cover it (at least one).
__device__ __forceinline__ int compacted_rank(const float* Dc) {
  int r = 0;
  while (r < RP && Dc[r] != 0.f) ++r;
  return r;
}
__device__ __forceinline__ int rank_kblocks(int r) { return r > 0 ? (r + 15) >> 4 : 1; }

// Stages whose x boxes a forward kernel requests before its dependency wait.
template <typename Args>
__device__ __forceinline__ int fwd_prefetched(const Args& p, int nstage) {
  if (!p.prefetch_x || (int)blockIdx.x >= p.ntiles) return 0;
  return p.nN < nstage ? p.nN : nstage;
}

__device__ void zero_tail_rows(uint8_t* stages, int nstage, uint8_t* zp_tile, int tt) {
  if (tt >= TILE) return;
  const int per_box = (TILE - tt) * 8;  // 16-byte units
  const int nbox = 2 * nstage + 1;
  for (int i = threadIdx.x; i < nbox * per_box; i += blockDim.x) {
    const int b = i / per_box, o = i - b * per_box;
    uint8_t* bp = b < 2 * nstage ? stages + (b >> 1) * STAGE + (b & 1) * BOX : zp_tile;
    *reinterpret_cast<uint4*>(bp + tt * 128 + o * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_async_smem();  // the MMAs read these rows through the async proxy
}

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ void tmem_alloc(uint32_t* slot) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   su32(slot)),
               "r"(TMEM_COLS)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ void tmem_free(uint32_t base) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base),
               "r"(TMEM_COLS)
               : "memory");
}

// ==========================================================================
// forward: y = ((x A) diag(Dc)) B per tile of up to 128 tokens
// (F8: x in E4M3, widened in shared memory by the converter warps)
// ==========================================================================
template <bool F8>
__global__ void __launch_bounds__(F8 ? NTHREADS_F8 : NTHREADS, 1)
    tt_fwd_kernel(const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_anr,
                  const __grid_constant__ CUtensorMap tm_bm,
                  const __grid_constant__ CUtensorMap tm_y,
                  const __grid_constant__ CUtensorMap tm_y16,
                  const __grid_constant__ CUtensorMap tm_zs, FwdArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1k(smem_raw);
  uint8_t* stages = base;
  uint8_t* zp_tile = base + NSTAGE_F * STAGE;
  uint8_t* staging = zp_tile + BOX;  // 2 boxes per epilogue warp
  SmemCommon& S = *reinterpret_cast<SmemCommon*>(staging + NEPI * 2 * STG);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) TL_STAMP(0, 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE_F; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.z_full, 1);
    mbar_init(&S.z_empty, NEPI);
    mbar_init(&S.zp_full, NEPI);
    mbar_init(&S.zp_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.x_full[b], 1);
      mbar_init(&S.x_empty[b], NEPI);
    }
    for (int s = 0; s < NSTAGE_F; ++s) mbar_init(&S.conv[s], NCONV);
    mbar_init(&S.fin, 1);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // x of the first tile's first chunks (rows 0..tt-1 of the activation
    // boxes; zero_tail_rows below writes the other rows)
    for (int s = 0; s < fwd_prefetched(p, NSTAGE_F); ++s) {
      uint8_t* st = stages + s * STAGE;
      const uint32_t act_bytes = (uint32_t)p.tt * 128;
      const int tok0 = blockIdx.x * p.tt;
      if (F8) {
        mbar_expect_tx(&S.full[s], act_bytes + BOX);
        tma_load(st + BOX, &tm_x, &S.full[s], s * CH, tok0);
      } else {
        mbar_expect_tx(&S.full[s], 2 * act_bytes + BOX);
        tma_load(st, &tm_x, &S.full[s], s * CH, tok0);
        tma_load(st + BOX, &tm_x, &S.full[s], s * CH + 64, tok0);
      }
    }
  }
  if (warp == 1) tmem_alloc(&S.tmem_base);
  pdl_wait();  // nothing a previous grid writes is touched before this point (but x above)
  pdl_trigger();
  if (threadIdx.x < RP) S.Dc[threadIdx.x] = p.Dc[threadIdx.x];
  zero_tail_rows(stages, NSTAGE_F, zp_tile, p.tt);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  if (threadIdx.x == 0) TL_STAMP(0, 1);
  volatile int* abort_flag = &S.abort_flag;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      int it = 0;
      int last_parity[NSTAGE_F];
      for (int s = 0; s < NSTAGE_F; ++s) last_parity[s] = -1;
      bool ok = true;
      const uint32_t act_bytes = (uint32_t)p.tt * 128;  // one activation box of tt rows
      // test hook: the first CTA leaves its first stage unloaded
      const bool skip_first = blockIdx.x == 0 && debug_take(TT_DEBUG_FWD_TOKENS);
      const int npre = fwd_prefetched(p, NSTAGE_F);  // x already requested
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x) {
        const int tok0 = tile * p.tt;
        for (int c = 0; ok && c < p.nN + p.nM; ++c, ++it) {
          const int s = it % NSTAGE_F;
          const uint32_t ph = (it / NSTAGE_F) & 1;
          if (!wait_bar(&S.empty[s], ph ^ 1, abort_flag, 1)) { ok = false; break; }
          if (skip_first && it == 0) continue;
          uint8_t* st = stages + s * STAGE;
          if (it < npre) {
            tma_load(st + OPND, &tm_anr, &S.full[s], 0, c * CH);
          } else if (c < p.nN) {
            if (F8) {  // one E4M3 box of 128 columns into the second bf16 box's bytes
              mbar_expect_tx(&S.full[s], act_bytes + BOX);
              tma_load(st + BOX, &tm_x, &S.full[s], c * CH, tok0);
            } else {
              mbar_expect_tx(&S.full[s], 2 * act_bytes + BOX);
              tma_load(st, &tm_x, &S.full[s], c * CH, tok0);
              tma_load(st + BOX, &tm_x, &S.full[s], c * CH + 64, tok0);
            }
            tma_load(st + OPND, &tm_anr, &S.full[s], 0, c * CH);  // [128 features][64 ranks]
          } else {
            mbar_expect_tx(&S.full[s], BOX);
            // [64 ranks][128 outputs] as two boxes of 64 outputs
            tma_load(st + OPND, &tm_bm, &S.full[s], (c - p.nN) * CH, 0);
            tma_load(st + OPND + BOX / 2, &tm_bm, &S.full[s], (c - p.nN) * CH + 64, 0);
          }
          last_parity[s] = (int)ph;
        }
      }
      for (int s = 0; s < NSTAGE_F; ++s)
        if (last_parity[s] >= 0) drain_bar(&S.full[s], (uint32_t)last_parity[s]);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_z = idesc(128, 64, 0, 1);   // B = Anr rows, MN-major
      const uint32_t id_y = idesc(128, 128, 0, 1);  // B = Bm rows, MN-major
      const uint32_t zp_addr = su32(zp_tile);
      uint64_t* ready = F8 ? S.conv : S.full;  // a stage the MMAs may read
      const int kb = rank_kblocks(compacted_rank(S.Dc));  // z' columns past r' are 0
      int it = 0, yc = 0, tl = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x, ++tl) {
        if (!wait_bar(&S.z_empty, (tl & 1) ^ 1, abort_flag, 2)) break;
        tc_fence_after();
        for (int c = 0; c < p.nN; ++c, ++it) {
          const int s = it % NSTAGE_F;
          if (!wait_bar(&ready[s], (it / NSTAGE_F) & 1, abort_flag, 3)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma(tmem + F_Z, kdesc(st + b * BOX) + 2 * k,
                  mndesc(st + OPND + b * (BOX / 2), 1024) + 128 * k, id_z, (c | b | k) != 0);
          mma_commit(&S.empty[s]);
        }
        if (!ok) break;
        mma_commit(&S.z_full);
        TL_STAMP(0, 2);
        if (!wait_bar(&S.zp_full, tl & 1, abort_flag, 4)) break;
        tc_fence_after();
        if (p.save_z) {  // keep z' for the backward (rows past T are clipped)
          tma_store(&tm_zs, zp_tile, 0, tile * p.tt);
          bulk_commit();
        }
        for (int c = 0; c < p.nM; ++c, ++it, ++yc) {
          const int s = it % NSTAGE_F;
          const int yb = yc & 1;
          if (!wait_bar(&S.x_empty[yb], ((yc >> 1) & 1) ^ 1, abort_flag, 5)) { ok = false; break; }
          if (c < 3) TL_STAMP(0, 13 + c);  // y buffer free
          if (!wait_bar(&ready[s], (it / NSTAGE_F) & 1, abort_flag, 6)) { ok = false; break; }
          if (c < 3) TL_STAMP(0, 10 + c);  // Bm chunk in shared memory
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
          for (int k = 0; k < kb; ++k)
            mma(tmem + F_Y + yb * 128, kdesc(zp_addr) + 2 * k,
                mndesc(st + OPND, BOX / 2) + 128 * k, id_y, k != 0);
          mma_commit(&S.empty[s]);
          mma_commit(&S.x_full[yb]);
        }
        if (!ok) break;
        if (p.save_z) bulk_wait_read<0>();  // the z' store has read the tile
        mma_commit(&S.zp_empty);
        TL_STAMP(0, 4);
      }
      if (p.save_z) bulk_wait_all();
      mma_commit(&S.fin);
      drain_bar(&S.fin, 0);
    }
  } else if (F8 && warp >= 2 + NEPI) {
    // ---------------- converters: every chunk in the producer's order; x
    // chunks are widened, operand-only chunks just pass through
    const int cw = warp - 2 - NEPI;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x) {
      for (int c = 0; c < p.nN + p.nM; ++c, ++it) {
        const int s = it % NSTAGE_F;
        if (!warp_wait(&S.full[s], (it / NSTAGE_F) & 1, abort_flag, 40)) { ok = false; break; }
        if (c < p.nN) {
          widen_e4m3_tile(stages + s * STAGE, cw, lane);
          fence_async_smem();
          __syncwarp();
        }
        if (lane == 0) mbar_arrive(&S.conv[s]);
      }
    }
  } else {
    // ---------------- epilogue: 8 warps, thread = (token row, column half)
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int row = 32 * q + lane;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    uint8_t* my_stg = staging + (warp - 2) * 2 * STG;
    int yc = 0, tl = 0;
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++tl) {
      float v[32];
      if (!warp_wait(&S.z_full, tl & 1, abort_flag, 7)) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_off + F_Z + 32 * h, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.z_empty);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= S.Dc[32 * h + j];
      if (!warp_wait(&S.zp_empty, (tl & 1) ^ 1, abort_flag, 8)) break;
      st_tile_half(zp_tile, row, h, v);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.zp_full);
      if (warp == 2 && lane == 0) TL_STAMP(0, 3);
      bool ok = true;
      for (int c = 0; c < p.nM; ++c, ++yc) {
        const int yb = yc & 1;
        if (!warp_wait(&S.x_full[yb], (yc >> 1) & 1, abort_flag, 9)) { ok = false; break; }
        if (warp == 2 && lane == 0 && c < 3) TL_STAMP(0, 7 + c);  // y chunk in TMEM
        tc_fence_after();
        uint8_t* box = my_stg + (yc & 1) * STG;
        if (lane == 0) bulk_wait_read<1>();  // the store that used this box is done reading
        __syncwarp();
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {
          tmem_ld32(tmem + lane_off + F_Y + yb * 128 + 64 * h + 32 * piece, v);
          stage_bf16_32(box, lane, piece, v);
        }
        tc_fence_before();
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&S.x_empty[yb]);
          const int col = c * CH + 64 * h;
          const int vq = p.tt - 32 * q;  // rows of this quadrant inside the tile
          if (col < p.M && vq > 0 && (int64_t)tile * p.tt + 32 * q < p.T)
            tma_store(vq >= 32 ? &tm_y : &tm_y16, box, col, tile * p.tt + 32 * q);
          bulk_commit();  // one group per chunk, empty if skipped: keeps the box ring in step
        }
      }
      if (!ok) break;
      if (warp == 2 && lane == 0) TL_STAMP(0, 5);
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) TL_STAMP(0, 6);
  if (warp == 1) tmem_free(tmem);
}

// ==========================================================================
// backward: per tile of up to 128 tokens
//   A  z   = x A                          (x streamed, 128 features a chunk;
//                                          skipped when the forward's z' is kept)
//   B  dz' = dy Bm^T ; dB^T += dy^T z'    (dy streamed, 128 outputs a chunk)
//   C  dx  = dz Anr^T ; dA += x^T dz      (x streamed again)
// with z' = z diag(Dc), dz = dz' diag(Dc), dDc += sum_t z * dz'.
// (F8: x and dy in E4M3, widened in shared memory by the converter warps)
// ==========================================================================
template <bool F8>
__global__ void __launch_bounds__(F8 ? NTHREADS_F8 : NTHREADS, 1)
    tt_bwd_kernel(const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_dy,
                  const __grid_constant__ CUtensorMap tm_bm,
                  const __grid_constant__ CUtensorMap tm_anr,
                  const __grid_constant__ CUtensorMap tm_dx,
                  const __grid_constant__ CUtensorMap tm_dx16,
                  const __grid_constant__ CUtensorMap tm_dac,
                  const __grid_constant__ CUtensorMap tm_dbc,
                  const __grid_constant__ CUtensorMap tm_zs, BwdArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align1k(smem_raw);
  uint8_t* stages = base;
  // z' (read by the phase-B MMAs) and dz (read by the phase-C MMAs) share
  // one tile: dz is written once phase B's MMAs are done, the next tile's z'
  // once phase C's are done
  uint8_t* zp_tile = base + NSTAGE_B * STAGE;
  uint8_t* dz_tile = zp_tile;
  uint8_t* staging = zp_tile + BOX;  // two boxes per epilogue warp
  SmemCommon& S = *reinterpret_cast<SmemCommon*>(staging + NEPI * 2 * STG);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) TL_STAMP(1, 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE_B; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.z_full, 1);
    mbar_init(&S.z_empty, NEPI);
    mbar_init(&S.zp_full, NEPI);
    mbar_init(&S.zp_empty, 1);
    mbar_init(&S.dzp_full, 1);
    mbar_init(&S.dzp_empty, NEPI);
    mbar_init(&S.dz_full, NEPI);
    mbar_init(&S.dz_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.w_full[b], 1);
      mbar_init(&S.w_empty[b], NEPI);
      mbar_init(&S.x_full[b], 1);
      mbar_init(&S.x_empty[b], NEPI);
    }
    for (int s = 0; s < NSTAGE_B; ++s) mbar_init(&S.conv[s], NCONV);
    mbar_init(&S.zl_full, 1);
    mbar_init(&S.fin, 1);
    S.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(&S.tmem_base);
  pdl_wait();  // nothing a previous grid writes is touched before this point
  pdl_trigger();
  if (threadIdx.x < RP) S.Dc[threadIdx.x] = p.Dc[threadIdx.x];
  zero_list(p.zero);
  zero_tail_rows(stages, NSTAGE_B, zp_tile, p.tt);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  if (threadIdx.x == 0) TL_STAMP(1, 1);
  volatile int* abort_flag = &S.abort_flag;
  const int nchunks = 2 * p.nN + p.nM;
  // with the forward's z' kept, phase A (x A) is skipped: chunks start at B
  const int cfirst = p.use_z ? p.nN : 0;

  if (warp == 0) {
    // ---------------- TMA producer: (z' tile,) A chunks, B chunks, C chunks per tile
    if (lane == 0) {
      int it = 0, tl = 0;
      int last_parity[NSTAGE_B];
      for (int s = 0; s < NSTAGE_B; ++s) last_parity[s] = -1;
      bool ok = true;
      const uint32_t act_bytes = (uint32_t)p.tt * 128;  // one activation box of tt rows
      // test hook: the first CTA leaves its first stage unloaded
      const bool skip_first = blockIdx.x == 0 && debug_take(TT_DEBUG_BWD_TOKENS);
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x, ++tl) {
        const int tok0 = tile * p.tt;
        if (p.use_z) {
          // the shared z'/dz tile is free once the previous tile's phase C is done
          if (!wait_bar(&S.dz_empty, (tl & 1) ^ 1, abort_flag, 30)) break;
          mbar_expect_tx(&S.zl_full, act_bytes);
          tma_load(zp_tile, &tm_zs, &S.zl_full, 0, tok0);
        }
        for (int c = cfirst; c < nchunks; ++c, ++it) {
          const int s = it % NSTAGE_B;
          const uint32_t ph = (it / NSTAGE_B) & 1;
          if (!wait_bar(&S.empty[s], ph ^ 1, abort_flag, 11)) { ok = false; break; }
          if (tl == 0) TLK(it);  // stage free, load issued
          if (skip_first && it == 0) continue;
          uint8_t* st = stages + s * STAGE;
          mbar_expect_tx(&S.full[s], (F8 ? act_bytes : 2 * act_bytes) + BOX);
          // activation tile: E4M3 as one box into the second bf16 box's bytes
          const bool is_dy = c >= p.nN && c < p.nN + p.nM;
          const CUtensorMap* act = is_dy ? &tm_dy : &tm_x;
          const int col = (c < p.nN      ? c
                           : is_dy       ? rot_chunk(c - p.nN, p.nM, tile)
                                         : rot_chunk(c - p.nN - p.nM, p.nN, tile)) *
                          CH;
          if (F8) {
            tma_load(st + BOX, act, &S.full[s], col, tok0);
          } else {
            tma_load(st, act, &S.full[s], col, tok0);
            tma_load(st + BOX, act, &S.full[s], col + 64, tok0);
          }
          if (c < p.nN) {  // A: Anr rows of the chunk, read MN-major
            tma_load(st + OPND, &tm_anr, &S.full[s], 0, col);
          } else if (is_dy) {  // B
            tma_load(st + OPND, &tm_bm, &S.full[s], col, 0);
            tma_load(st + OPND + BOX / 2, &tm_bm, &S.full[s], col + 64, 0);
          } else {  // C
            tma_load(st + OPND, &tm_anr, &S.full[s], 0, col);
          }
          last_parity[s] = (int)ph;
        }
      }
      for (int s = 0; s < NSTAGE_B; ++s)
        if (last_parity[s] >= 0) drain_bar(&S.full[s], (uint32_t)last_parity[s]);
      if (p.use_z && tl > 0) drain_bar(&S.zl_full, (uint32_t)((tl - 1) & 1));
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      // dz' = dy Bm^T needs only the compacted ranks: N = 32 when r' <= 32
      // (Bm rows past r' are zero); dx = dz Anr^T only the K blocks that cover r'
      const int rprime = compacted_rank(S.Dc);
      const int kb = rank_kblocks(rprime);
      const uint32_t id_r = idesc(128, rprime <= 32 ? 32 : 64, 0, 0);  // token x rank, K-major
      const uint32_t id_a = idesc(128, 64, 0, 1);     // token x rank, B = Anr rows MN-major
      const uint32_t id_w = idesc(128, 64, 1, 1);     // weight x rank, MN-major
      const uint32_t id_x = idesc(128, 128, 0, 0);    // token x feature, K-major
      const uint32_t zp_addr = su32(zp_tile);
      const uint32_t dz_addr = su32(dz_tile);
      uint64_t* ready = F8 ? S.conv : S.full;  // a stage the MMAs may read
      int it = 0, wc = 0, xc = 0, tl = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x, ++tl) {
        // A: z = x A
        if (!p.use_z && !wait_bar(&S.z_empty, (tl & 1) ^ 1, abort_flag, 12)) break;
        tc_fence_after();
        for (int c = 0; c < p.nN && !p.use_z; ++c, ++it) {
          const int s = it % NSTAGE_B;
          if (!wait_bar(&ready[s], (it / NSTAGE_B) & 1, abort_flag, 13)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma(tmem + B_Z, kdesc(st + b * BOX) + 2 * k,
                  mndesc(st + OPND + b * (BOX / 2), 1024) + 128 * k, id_a, (c | b | k) != 0);
          mma_commit(&S.empty[s]);
        }
        if (!ok) break;
        if (!p.use_z) mma_commit(&S.z_full);
        TL_STAMP(1, 2);
        // B: dz' = dy Bm^T, dB^T chunk = dy^T z'
        if (!wait_bar(&S.dzp_empty, (tl & 1) ^ 1, abort_flag, 14)) break;
        tc_fence_after();
        for (int c = 0; c < p.nM; ++c, ++it, ++wc) {
          const int s = it % NSTAGE_B;
          if (!wait_bar(&ready[s], (it / NSTAGE_B) & 1, abort_flag, 15)) { ok = false; break; }
          if (tl == 0) TLK(2 * c);  // dy chunk c in shared memory
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
#pragma unroll
          for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma(tmem + B_DZP, kdesc(st + b * BOX) + 2 * k,
                  kdesc(st + OPND + b * (BOX / 2)) + 2 * k, id_r, (c | b | k) != 0);
          if (c == 0) {  // z' written by the epilogue, or loaded from the forward's copy
            if (!wait_bar(p.use_z ? &S.zl_full : &S.zp_full, tl & 1, abort_flag, 16)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const int wb = wc & 1;
          if (!wait_bar(&S.w_empty[wb], ((wc >> 1) & 1) ^ 1, abort_flag, 17)) { ok = false; break; }
          if (tl == 0) TLK(2 * c + 1);  // W buffer free
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma(tmem + B_W + wb * 64, mndesc(st, BOX) + 128 * k, mndesc(zp_addr, 1024) + 128 * k,
                id_w, k != 0);
          mma_commit(&S.w_full[wb]);
          mma_commit(&S.empty[s]);
        }
        if (!ok) break;
        mma_commit(&S.dzp_full);
        TL_STAMP(1, 4);
        mma_commit(&S.zp_empty);
        // C: dx = dz Anr^T, dA chunk = x^T dz
        if (!wait_bar(&S.dz_full, tl & 1, abort_flag, 18)) break;
        tc_fence_after();
        for (int c = 0; c < p.nN; ++c, ++it, ++xc, ++wc) {
          const int s = it % NSTAGE_B;
          if (!wait_bar(&ready[s], (it / NSTAGE_B) & 1, abort_flag, 19)) { ok = false; break; }
          const int xb = xc & 1;
          if (!wait_bar(&S.x_empty[xb], ((xc >> 1) & 1) ^ 1, abort_flag, 20)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = su32(stages + s * STAGE);
          for (int k = 0; k < kb; ++k)
            mma(tmem + B_X + xb * 128, kdesc(dz_addr) + 2 * k, kdesc(st + OPND) + 2 * k, id_x,
                k != 0);
          mma_commit(&S.x_full[xb]);
          const int wb = wc & 1;
          if (!wait_bar(&S.w_empty[wb], ((wc >> 1) & 1) ^ 1, abort_flag, 21)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma(tmem + B_W + wb * 64, mndesc(st, BOX) + 128 * k, mndesc(dz_addr, 1024) + 128 * k,
                id_w, k != 0);
          mma_commit(&S.w_full[wb]);
          mma_commit(&S.empty[s]);
        }
        if (!ok) break;
        mma_commit(&S.dz_empty);
      }
      mma_commit(&S.fin);
      drain_bar(&S.fin, 0);
    }
  } else if (F8 && warp >= 2 + NEPI) {
    // ---------------- converters: every chunk (x, dy, x) in the producer's order
    const int cw = warp - 2 - NEPI;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.ntiles; tile += gridDim.x) {
      for (int c = cfirst; c < nchunks; ++c, ++it) {
        const int s = it % NSTAGE_B;
        if (!warp_wait(&S.full[s], (it / NSTAGE_B) & 1, abort_flag, 41)) { ok = false; break; }
        widen_e4m3_tile(stages + s * STAGE, cw, lane);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.conv[s]);
      }
    }
  } else {
    // ---------------- epilogue
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int row = 32 * q + lane;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const int rprime = p.rinfo[0];
    uint8_t* my_stg = staging + (warp - 2) * 2 * STG;
    int nst = 0;  // bulk operations this warp issued: they alternate between its two boxes
    int wc = 0, xc = 0, tl = 0;
    for (int tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x, ++tl) {
      float z[32], v[32];
      bool ok = true;
      if (!p.use_z) {
        // E1: z -> z' tile
        if (!warp_wait(&S.z_full, tl & 1, abort_flag, 22)) break;
        tc_fence_after();
        tmem_ld32(tmem + lane_off + B_Z + 32 * h, z);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.z_empty);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = z[j] * S.Dc[32 * h + j];
        // the shared z'/dz tile is free once the previous tile's phase C is done
        if (!warp_wait(&S.dz_empty, (tl & 1) ^ 1, abort_flag, 23)) break;
        st_tile_half(zp_tile, row, h, v);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.zp_full);
      }
      if (warp == 2 && lane == 0) TL_STAMP(1, 3);
      // E2: dB^T chunks (row = output index within the chunk)
      for (int c = 0; c < p.nM; ++c, ++wc) {
        const int wb = wc & 1;
        if (!warp_wait(&S.w_full[wb], (wc >> 1) & 1, abort_flag, 24)) { ok = false; break; }
        if (tl == 0) TLK(2 * c);  // W chunk c in TMEM
        tc_fence_after();
        tmem_ld32(tmem + lane_off + B_W + wb * 64 + 32 * h, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.w_empty[wb]);
        if (tl == 0) TLK(2 * c + 1);  // released
        // rows = outputs c*128 + 32q.., columns = compacted ranks 32h..
        const int cb = rot_chunk(c, p.nM, tile);  // the producer's order of dy chunks
        if (32 * h < rprime && cb * CH + 32 * q < p.M) {
          uint8_t* box = my_stg + (nst & 1) * STG;
          if (lane == 0) bulk_wait_read<1>();  // the operation that used this box is done reading
          __syncwarp();
          stage_f32_32(box, lane, v);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (p.det && tl == 0)
              tma_store(&tm_dbc, box, 32 * h, blockIdx.x * p.M + cb * CH + 32 * q);
            else
              tma_reduce_add(&tm_dbc, box, 32 * h,
                             (p.det ? blockIdx.x * p.M : 0) + cb * CH + 32 * q);
            bulk_commit();
          }
          ++nst;
        }
      }
      if (!ok) break;
      // E3: dz' -> dDc, dz tile (columns 32.. are not computed when r' <= 32)
      if (!warp_wait(&S.dzp_full, tl & 1, abort_flag, 25)) break;
      if (tl == 0) TLK(20);
      tc_fence_after();
      tmem_ld32(tmem + lane_off + B_DZP + 32 * h, v);
      if (32 * h >= rprime) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.dzp_empty);
      if (p.use_z) {
        // z' of this thread's row from the loaded tile (read before dz
        // overwrites the same bytes below); sum z' dz' / Dc = sum z dz'
        if (!warp_wait(&S.zl_full, tl & 1, abort_flag, 31)) break;
        ld_tile_half(zp_tile, row, h, z);
      }
      {
        float pr[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) pr[j] = z[j] * v[j];
        float colsum = warp_transpose_sum(pr, lane);
        if (32 * h + lane < rprime) {
          if (p.use_z) colsum = colsum / S.Dc[32 * h + lane];  // nonzero: compacted column
          if (p.det) {  // this lane alone owns the entry of its CTA and quadrant
            float* e = p.dDslot + ((size_t)blockIdx.x * 4 + q) * RP + 32 * h + lane;
            *e = tl == 0 ? colsum : *e + colsum;
          } else {
            atomicAdd(p.dDc + 32 * h + lane, colsum);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= S.Dc[32 * h + j];
      // phase B's MMAs (readers of z' in the shared tile) are done
      if (!warp_wait(&S.zp_empty, tl & 1, abort_flag, 26)) break;
      st_tile_half(dz_tile, row, h, v);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.dz_full);
      if (tl == 0) TLK(21);
      if (warp == 2 && lane == 0) TL_STAMP(1, 5);
      // E4: dx chunks (row = token), dA chunks (row = feature within the chunk)
      for (int c = 0; c < p.nN; ++c, ++xc, ++wc) {
        const int xb = xc & 1;
        if (!warp_wait(&S.x_full[xb], (xc >> 1) & 1, abort_flag, 27)) { ok = false; break; }
        if (tl == 0) TLK(22 + 2 * c);  // dx chunk c in TMEM
        tc_fence_after();
        const int cx = rot_chunk(c, p.nN, tile);  // the producer's order of phase-C x chunks
        const int col = cx * CH + 64 * h;
        const int vq = p.tt - 32 * q;  // rows of this quadrant inside the tile
        const bool st_dx = col < p.N && vq > 0 && (int64_t)tile * p.tt + 32 * q < p.T;
        uint8_t* box = my_stg + (nst & 1) * STG;
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {
          tmem_ld32(tmem + lane_off + B_X + xb * 128 + 64 * h + 32 * piece, v);
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
        if (st_dx) ++nst;
        const int wb = wc & 1;
        if (!warp_wait(&S.w_full[wb], (wc >> 1) & 1, abort_flag, 28)) { ok = false; break; }
        tc_fence_after();
        tmem_ld32(tmem + lane_off + B_W + wb * 64 + 32 * h, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.w_empty[wb]);
        // rows = features c*128 + 32q.., columns = compacted ranks 32h..
        if (32 * h < rprime && cx * CH + 32 * q < p.N) {
          uint8_t* box2 = my_stg + (nst & 1) * STG;
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          stage_f32_32(box2, lane, v);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (p.det && tl == 0)
              tma_store(&tm_dac, box2, 32 * h, blockIdx.x * p.N + cx * CH + 32 * q);
            else
              tma_reduce_add(&tm_dac, box2, 32 * h,
                             (p.det ? blockIdx.x * p.N : 0) + cx * CH + 32 * q);
            bulk_commit();
          }
          ++nst;
        }
      }
      if (!ok) break;
      // the next tile's adds into this CTA's slot come after this tile's
      if (p.det && lane == 0) bulk_wait_all();
      if (warp == 2 && lane == 0) TL_STAMP(1, 6);
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) TL_STAMP(1, 7);
  if (warp == 1) tmem_free(tmem);
}

// ==========================================================================
// fixed-order sum of the per-CTA token-sum slots (TT_DETERMINISTIC)
//   dAc[i] = sum_k slotA[k][i], dBc[i] = sum_k slotB[k][i],
//   dDc[c] = sum_{k, q} slotD[k][q][c]
// The slots of one output are split into four fixed ranges of k; each range
// is summed in increasing k by its own quarter of the block (eight slots in
// flight a thread, four floats a load), and the four partial sums are added
// in range order: the same order, and so the same bits, on every call.
// Columns at or past `wcol` of a 64-wide row (ranks the layer does not have:
// the token kernel writes no slot entry there) come out 0 without a read.
// ==========================================================================
__device__ __forceinline__ void add4(float4& s, const float4 v) {
  s.x += v.x;
  s.y += v.y;
  s.z += v.z;
  s.w += v.w;
}

constexpr int kDetCols = 64;  // float4 columns a block handles at a time (x 4 ranges = 256 threads)

__global__ void __launch_bounds__(4 * kDetCols) det_sum_kernel(
    const float* __restrict__ slotA, const float* __restrict__ slotB,
    const float* __restrict__ slotD, int G, int64_t nA, int64_t nB, int wcol, float* dAc,
    float* dBc, float* dDc) {
  pdl_wait();  // the token kernel's slots are complete
  pdl_trigger();
  __shared__ float4 part[4][kDetCols];
  const int kg = (int)threadIdx.x / kDetCols, vc = (int)threadIdx.x % kDetCols;
  const int64_t nvA = nA / 4, nvB = nB / 4, nvD = RP / 4, nv = nvA + nvB + nvD;
  for (int64_t v0 = (int64_t)blockIdx.x * kDetCols; v0 < nv; v0 += (int64_t)gridDim.x * kDetCols) {
    const int64_t v = v0 + vc;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* base = nullptr;
    int64_t stride = 0;  // float4s from one slot to the next
    int cnt = 0;         // slots summed (0: a column past wcol)
    if (4 * (int)(v % (RP / 4)) >= wcol) {
      // nA and nB are whole 64-wide rows, so v % 16 is the column in every region
    } else if (v < nvA) {
      base = reinterpret_cast<const float4*>(slotA) + v;
      stride = nvA;
      cnt = G;
    } else if (v < nvA + nvB) {
      base = reinterpret_cast<const float4*>(slotB) + (v - nvA);
      stride = nvB;
      cnt = G;
    } else if (v < nv) {
      base = reinterpret_cast<const float4*>(slotD) + (v - nvA - nvB);
      stride = nvD;  // slots (k, q) in k-major order
      cnt = 4 * G;
    }
    const int k0 = (int)((int64_t)cnt * kg / 4), k1 = (int)((int64_t)cnt * (kg + 1) / 4);
    int k = k0;
    for (; k + 8 <= k1; k += 8) {
      float4 r[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) r[j] = __ldcg(base + (int64_t)(k + j) * stride);
#pragma unroll
      for (int j = 0; j < 8; ++j) add4(s, r[j]);
    }
    for (; k < k1; ++k) add4(s, __ldcg(base + (int64_t)k * stride));
    part[kg][vc] = s;
    __syncthreads();
    if (kg == 0 && v < nv) {
      float4 t = part[0][vc];
      add4(t, part[1][vc]);
      add4(t, part[2][vc]);
      add4(t, part[3][vc]);
      float* out = v < nvA ? dAc + 4 * v : v < nvA + nvB ? dBc + 4 * (v - nvA) : dDc + 4 * (v - nvA - nvB);
      out[0] = t.x;
      out[1] = t.y;
      out[2] = t.z;
      out[3] = t.w;
    }
    __syncthreads();
  }
}

// ==========================================================================
// operand packing (compaction of the middle rank) and gradient unpacking,
// run as units of the merge engine
// ==========================================================================
constexpr int kPackPer = 4096;      // elements per engine unit, unless the phase balancing widens it
constexpr int kPackPerMax = 16384;  // the widest unit the balancing makes

// Compaction of the middle rank, computed by the whole block in parallel:
// pos[a] = position of a among the nonzero entries of D (or -1), kept[c] = a
// for c < r' (-1 beyond), *rcount = r'.  All threads must call it.
__device__ void compaction_map(const float* __restrict__ D, int rd, int* pos, int* kept,
                               int* rcount) {
  __shared__ unsigned masks[2];
  __syncthreads();
  const int a = threadIdx.x;
  bool nz = false;
  if (a < RP) {
    nz = a < rd && __ldcg(D + a) != 0.f;
    const unsigned m = __ballot_sync(0xffffffffu, nz);
    if ((a & 31) == 0) masks[a >> 5] = m;
  }
  __syncthreads();
  if (a < RP) {
    const unsigned m0 = masks[0], m1 = masks[1];
    const int before = a < 32 ? __popc(m0 & ((1u << a) - 1u))
                              : __popc(m0) + __popc(m1 & ((1u << (a - 32)) - 1u));
    const int r = __popc(m0) + __popc(m1);
    if (pos) pos[a] = nz ? before : -1;
    if (kept) {
      if (nz) kept[before] = a;
      if (a >= r) kept[a] = -1;
    }
    if (a == 0 && rcount) *rcount = r;
  }
  __syncthreads();
}

// pad_only: write only the padding columns (c >= r') and the metadata; the
// merge GEMMs' epilogues write the compacted columns themselves.
__device__ void tc_pack_unit(const float* __restrict__ A, const float* __restrict__ B,
                             const float* __restrict__ Dmid, int rd, int N, int M,
                             const TcPtrs& p, int zero_grads, int pad_only, int chunk, int unit) {
  __shared__ int kept[RP];
  __shared__ int rcount;
  compaction_map(Dmid, rd, nullptr, kept, &rcount);
  const int64_t nA = (int64_t)N * RP, nB = (int64_t)M * RP;
  __nv_bfloat16* Anr = static_cast<__nv_bfloat16*>(p.Anr);
  __nv_bfloat16* Bm = static_cast<__nv_bfloat16*>(p.Bm);
  for (int e = threadIdx.x; e < chunk; e += blockDim.x) {
    const int64_t i = (int64_t)unit * chunk + e;
    if (i < nA) {
      const int j = (int)(i / RP), c = (int)(i % RP);
      if (!pad_only || kept[c] < 0) {
        const float v = kept[c] >= 0 ? __ldcg(A + (int64_t)j * rd + kept[c]) : 0.f;
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        Anr[i] = b;
      }
      if (zero_grads) p.dAc[i] = 0.f;
    } else if (i < nA + nB) {
      const int64_t k = i - nA;  // Bm [RP][M], walked in its own (row-major) order
      const int c = (int)(k / M), o = (int)(k - (int64_t)c * M);
      if (!pad_only || kept[c] < 0) {
        const float v = kept[c] >= 0 ? __ldcg(B + (int64_t)kept[c] * M + o) : 0.f;
        Bm[k] = __float2bfloat16_rn(v);
      }
      if (zero_grads) p.dBc[k] = 0.f;  // dBc has the same size, [M][RP]
    } else if (i < nA + nB + RP) {
      const int c = (int)(i - nA - nB);
      p.Dc[c] = kept[c] >= 0 ? Dmid[kept[c]] : 0.f;
      p.rinfo[1 + c] = kept[c];
      if (c == 0) p.rinfo[0] = rcount;
      if (zero_grads) p.dDc[c] = 0.f;
    }
  }
}

// dD_d (uncompacted, prune convention, accumulate) from the token sum dDc.
__device__ void tc_dd_unit(const TcPtrs& p, const float* Dmid, int rd, float* dDout, int acc) {
  __shared__ int pos[RP];
  compaction_map(Dmid, rd, pos, nullptr, nullptr);
  if (threadIdx.x < rd) {
    const int a = threadIdx.x;
    const int c = pos[a];
    const float v = c >= 0 ? __ldcg(p.dDc + c) : 0.f;
    dDout[a] = acc ? dDout[a] + v : v;
  }
}

__device__ void tc_unpack_unit(const TcPtrs& p, const float* Dmid, int rd, int N, int M,
                               float* dA, float* dB, float* dDout, int acc, int chunk, int unit) {
  __shared__ int pos[RP];
  compaction_map(Dmid, rd, pos, nullptr, nullptr);
  const int64_t nA = (int64_t)N * rd, nB = (int64_t)rd * M;
  for (int e = threadIdx.x; e < chunk; e += blockDim.x) {
    const int64_t i = (int64_t)unit * chunk + e;
    if (i < nA) {
      const int j = (int)(i / rd), a = (int)(i % rd);
      dA[i] = pos[a] >= 0 ? __ldcg(p.dAc + (int64_t)j * RP + pos[a]) : 0.f;
    } else if (i < nA + nB) {
      const int64_t k = i - nA;
      const int a = (int)(k / M), o = (int)(k % M);
      dB[k] = pos[a] >= 0 ? __ldcg(p.dBc + (int64_t)o * RP + pos[a]) : 0.f;
    } else if (i < nA + nB + rd) {
      const int a = (int)(i - nA - nB);
      const float v = pos[a] >= 0 ? __ldcg(p.dDc + pos[a]) : 0.f;
      dDout[a] = acc ? dDout[a] + v : v;
    }
  }
}

// ==========================================================================
// host side
// ==========================================================================
struct TcLayout {
  size_t Anr, Bm, Dc, rinfo, dAc, dBc, dDc, total;
};

size_t al256(size_t v) { return (v + 255) / 256 * 256; }

TcLayout tc_layout(const LayerPlan& L) {
  TcLayout t;
  size_t o = 0;
  auto take = [&](size_t b) {
    size_t r = o;
    o = al256(o + b);
    return r;
  };
  t.Anr = take((size_t)L.N * RP * 2);
  t.Bm = take((size_t)RP * L.M * 2);
  t.Dc = take(RP * 4);
  t.rinfo = take((RP + 1) * 4);
  t.dAc = take((size_t)L.N * RP * 4);
  t.dBc = take((size_t)RP * L.M * 4);
  t.dDc = take(RP * 4);
  t.total = o;
  return t;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

enum MapType { kMapBF16, kMapF32, kMapU8 };

// 2-D tensor (outer x inner, row-major) of bf16, f32 or bytes (E4M3 codes),
// box (box_outer x box_inner), 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer, MapType type = kMapBF16) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t esz = type == kMapF32 ? 4 : type == kMapU8 ? 1 : 2;
  const CUtensorMapDataType dt = type == kMapF32  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : type == kMapU8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                  : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * esz};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

constexpr size_t kSmemFwd = NSTAGE_F * STAGE + BOX + NEPI * 2 * STG + sizeof(SmemCommon) + 1024;
constexpr size_t kSmemBwd = NSTAGE_B * STAGE + BOX + NEPI * 2 * STG + sizeof(SmemCommon) + 1024;
static_assert(kSmemFwd <= 227 * 1024, "forward smem");
static_assert(kSmemBwd <= 227 * 1024, "backward smem");

int num_sms() { return device_sms(); }

cudaError_t set_smem_attrs() {
  static PerDevice once;
  return once.get([] {
    const std::pair<const void*, size_t> k[4] = {
        {(const void*)tt_fwd_kernel<false>, kSmemFwd}, {(const void*)tt_fwd_kernel<true>, kSmemFwd},
        {(const void*)tt_bwd_kernel<false>, kSmemBwd}, {(const void*)tt_bwd_kernel<true>, kSmemBwd}};
    cudaError_t err = cudaSuccess;
    for (int i = 0; i < 4 && err == cudaSuccess; ++i)
      err = cudaFuncSetAttribute(k[i].first, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)k[i].second);
    return err;
  });
}

// Tokens per tile: the fewest tiles of at most TILE tokens that give every
// SM the same number of waves, rounded up to a multiple of 16 (16 .. TILE);
// but full TILE-token tiles when they make one wave over at least three
// quarters of the SMs: a tile's pass takes about as long at 112 tokens as at
// 128, and the SMs left idle take the next launch's first CTAs early.  At
// 16384 tokens on 152 SMs that is 128 tiles of 128 tokens (the balanced
// choice, 147 tiles of 112, made the 768 x 768 step 1.7 % slower).
// TTC_TILE_TOKENS (16 .. 128, multiple of 16) fixes it.
int tokens_per_tile(int64_t T) {
  static int forced = -1;
  if (forced < 0) {
    const char* e = getenv("TTC_TILE_TOKENS");
    const int v = e ? atoi(e) : 0;
    forced = (v >= 16 && v <= TILE && v % 16 == 0) ? v : 0;
  }
  if (forced) return forced;
  const int64_t sms = num_sms();
  const int64_t waves = (T + (int64_t)TILE * sms - 1) / ((int64_t)TILE * sms);
  if (waves == 1 && 4 * T >= 3 * (int64_t)TILE * sms) return TILE;
  int64_t tt = (T + waves * sms - 1) / (waves * sms);
  tt = (tt + 15) / 16 * 16;
  return (int)(tt < 16 ? 16 : tt > TILE ? TILE : tt);
}

// Programmatic dependent launch is on unless TTC_NO_PDL is set (to 1).
bool pdl_enabled() {
  static int on = -1;
  if (on < 0) {
    const char* e = getenv("TTC_NO_PDL");
    on = (e && e[0] && e[0] != '0') ? 0 : 1;
  }
  return on == 1;
}

// Launch with the programmatic-serialization attribute (and optionally as a
// cooperative grid).  The kernels call pdl_wait() before reading anything a
// predecessor may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                      bool cooperative, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  if (pdl_enabled()) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cooperative) {
    attrs[n].id = cudaLaunchAttributeCooperative;
    attrs[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace

bool tc_supported(const LayerPlan& L) {
  return L.rd <= RP && L.N % 8 == 0 && L.M % 8 == 0 && L.N >= CH && L.M >= CH &&
         L.N <= (1 << 20) && L.M <= (1 << 20);
}

bool tc_f8_supported(const LayerPlan& L) {
  return tc_supported(L) && L.N % 16 == 0 && L.M % 16 == 0;
}

size_t tc_operand_bytes(const LayerPlan& L) {
  return tc_supported(L) ? tc_layout(L).total : 256;
}

TcPtrs tc_ptrs(const LayerPlan& L, void* ws, size_t off) {
  const TcLayout t = tc_layout(L);
  TcPtrs p;
  p.Anr = at<void>(ws, off + t.Anr);
  p.Bm = at<void>(ws, off + t.Bm);
  p.Dc = at<float>(ws, off + t.Dc);
  p.rinfo = at<int>(ws, off + t.rinfo);
  p.dAc = at<float>(ws, off + t.dAc);
  p.dBc = at<float>(ws, off + t.dBc);
  p.dDc = at<float>(ws, off + t.dDc);
  return p;
}

tt_status tc_forward(const LayerPlan& L, int64_t T, const void* x, void* y, void* ws, size_t off,
                     bool f8, void* zs, bool prefetch_x, cudaStream_t st) {
  if (T <= 0) return TT_OK;
  if (T > (int64_t)0x7FFFFFFF - TILE) return TT_ERR_UNSUPPORTED;
  if (f8 && !tc_f8_supported(L)) return TT_ERR_UNSUPPORTED;
  const TcLayout t = tc_layout(L);
  if (set_smem_attrs() != cudaSuccess) return TT_ERR_CUDA;
  const int tt = tokens_per_tile(T);
  CUtensorMap mx, manr, mbm, my, my16, mzs;
  const bool mx_ok = f8 ? make_map(&mx, x, L.N, T, CH, tt, kMapU8) : make_map(&mx, x, L.N, T, 64, tt);
  if (!mx_ok ||
      !make_map(&manr, at<void>(ws, off + t.Anr), RP, L.N, 64, CH) ||
      !make_map(&mbm, at<void>(ws, off + t.Bm), L.M, RP, 64, RP) ||
      !make_map(&my, y, L.M, T, 64, 32) || !make_map(&my16, y, L.M, T, 64, 16) ||
      !make_map(&mzs, zs ? zs : y, RP, T, 64, tt))
    return TT_ERR_CUDA;
  FwdArgs a;
  a.T = T;
  a.N = (int)L.N;
  a.M = (int)L.M;
  a.nN = (int)((L.N + CH - 1) / CH);
  a.nM = (int)((L.M + CH - 1) / CH);
  a.tt = tt;
  a.ntiles = (int)((T + tt - 1) / tt);
  a.save_z = zs != nullptr;
  a.prefetch_x = prefetch_x && pdl_enabled() ? 1 : 0;
  a.Dc = at<float>(ws, off + t.Dc);
  a.y = static_cast<__nv_bfloat16*>(y);
  int grid = a.ntiles < num_sms() ? a.ntiles : num_sms();
  cudaError_t e =
      f8 ? launch_ex(tt_fwd_kernel<true>, grid, NTHREADS_F8, kSmemFwd, st, false, mx, manr, mbm, my,
                     my16, mzs, a)
         : launch_ex(tt_fwd_kernel<false>, grid, NTHREADS, kSmemFwd, st, false, mx, manr, mbm, my,
                     my16, mzs, a);
  count_launches(1);
  return e == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

cudaError_t zero_list_memset(const ZeroList& z, cudaStream_t st) {
  for (int r = 0; r < z.count; ++r) {
    cudaError_t e = cudaMemsetAsync(z.p[r], 0, (size_t)z.n[r] * sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// The fixed-order sums (TT_DETERMINISTIC) of one layer's token-sum slots,
// filled by the `grid` CTAs of a token pass, into its dAc, dBc and dDc.
cudaError_t det_sum_launch(const LayerPlan& L, const DetSlots& det, int grid, float* dAc,
                           float* dBc, float* dDc, cudaStream_t st) {
  const int64_t nA = L.N * RP, nB = L.M * RP;
  const int64_t cols = (nA + nB + RP) / 4;
  const int blocks = (int)((cols + kDetCols - 1) / kDetCols < 8 * num_sms()
                               ? (cols + kDetCols - 1) / kDetCols
                               : 8 * num_sms());
  const cudaError_t e = launch_ex(det_sum_kernel, blocks, 4 * kDetCols, 0, st, false,
                                  (const float*)det.a, (const float*)det.b, (const float*)det.d,
                                  grid, nA, nB, L.rd <= 32 ? 32 : RP, dAc, dBc, dDc);
  count_launches(1);
  return e;
}

tt_status tc_backward(const LayerPlan& L, int64_t T, const void* x, const void* dy, void* dx,
                      void* ws, size_t off, const ZeroList& zero, bool f8, const void* zs,
                      const DetSlots* det, cudaStream_t st) {
  if (f8 && !tc_f8_supported(L)) return TT_ERR_UNSUPPORTED;
  if (T <= 0) return zero_list_memset(zero, st) == cudaSuccess ? TT_OK : TT_ERR_CUDA;
  if (T > (int64_t)0x7FFFFFFF - TILE) return TT_ERR_UNSUPPORTED;
  const TcLayout t = tc_layout(L);
  if (set_smem_attrs() != cudaSuccess) return TT_ERR_CUDA;
  if (det && (det->count < 1 || (int64_t)det->count * (L.N > L.M ? L.N : L.M) > 0x7FFFFFFF))
    return TT_ERR_UNSUPPORTED;
  // a fixed summation order wants a fixed token blocking: 128-token tiles
  const int tt = det ? TILE : tokens_per_tile(T);
  CUtensorMap mx, mdy, mbm, manr, mdx, mdx16, mdac, mdbc, mzs;
  const bool act_ok = f8 ? make_map(&mx, x, L.N, T, CH, tt, kMapU8) &&
                               make_map(&mdy, dy, L.M, T, CH, tt, kMapU8)
                         : make_map(&mx, x, L.N, T, 64, tt) && make_map(&mdy, dy, L.M, T, 64, tt);
  if (!act_ok ||
      !make_map(&mbm, at<void>(ws, off + t.Bm), L.M, RP, 64, RP) ||
      !make_map(&manr, at<void>(ws, off + t.Anr), RP, L.N, 64, CH) ||
      !make_map(&mdx, dx, L.N, T, 64, 32) || !make_map(&mdx16, dx, L.N, T, 64, 16) ||
      !make_map(&mdac, det ? det->a : at<void>(ws, off + t.dAc), RP,
                L.N * (det ? det->count : 1), 32, 32, kMapF32) ||
      !make_map(&mdbc, det ? det->b : at<void>(ws, off + t.dBc), RP,
                L.M * (det ? det->count : 1), 32, 32, kMapF32) ||
      !make_map(&mzs, zs ? zs : dx, RP, T, 64, tt))
    return TT_ERR_CUDA;
  BwdArgs a;
  a.T = T;
  a.N = (int)L.N;
  a.M = (int)L.M;
  a.nN = (int)((L.N + CH - 1) / CH);
  a.nM = (int)((L.M + CH - 1) / CH);
  a.tt = tt;
  a.ntiles = (int)((T + tt - 1) / tt);
  a.Dc = at<float>(ws, off + t.Dc);
  a.rinfo = at<int>(ws, off + t.rinfo);
  a.dx = static_cast<__nv_bfloat16*>(dx);
  a.dAc = at<float>(ws, off + t.dAc);
  a.dBc = at<float>(ws, off + t.dBc);
  a.dDc = at<float>(ws, off + t.dDc);
  a.zero = zero;
  a.use_z = zs != nullptr;
  a.det = det ? 1 : 0;
  a.dDslot = det ? det->d : nullptr;
  int grid = a.ntiles < num_sms() ? a.ntiles : num_sms();
  if (det && grid > det->count) grid = det->count;
  cudaError_t e = f8 ? launch_ex(tt_bwd_kernel<true>, grid, NTHREADS_F8, kSmemBwd, st, false, mx,
                                 mdy, mbm, manr, mdx, mdx16, mdac, mdbc, mzs, a)
                      : launch_ex(tt_bwd_kernel<false>, grid, NTHREADS, kSmemBwd, st, false, mx, mdy,
                                  mbm, manr, mdx, mdx16, mdac, mdbc, mzs, a);
  count_launches(1);
  if (e != cudaSuccess) return TT_ERR_CUDA;
  if (det) {  // the slots of the `grid` CTAs, summed in CTA order
    e = det_sum_launch(L, *det, grid, a.dAc, a.dBc, a.dDc, st);
    if (e != cudaSuccess) return TT_ERR_CUDA;
  }
  return TT_OK;
}

}  // namespace ttc

extern "C" tt_status tt_set_wait_limit_ns(uint64_t ns) {
  if (ns < 1000) return TT_ERR_INVALID_ARG;
  const unsigned long long v = ns;
  return cudaMemcpyToSymbol(ttc::g_wait_limit_ns, &v, sizeof(v)) == cudaSuccess ? TT_OK
                                                                              : TT_ERR_CUDA;
}

extern "C" tt_status tt_debug_skip_arrival(int site) {
  if (site < 0 || site > TT_DEBUG_MERGE_BARRIER) return TT_ERR_INVALID_ARG;
  return cudaMemcpyToSymbol(ttc::g_debug_skip, &site, sizeof(site)) == cudaSuccess ? TT_OK
                                                                                  : TT_ERR_CUDA;
}

#include "merge_engine.cuh"
#include "ffn_fused.cuh"
#include "qkv_fused.cuh"

#ifdef TTC_TIMELINE
extern "C" int ttc_timeline_read(void* host, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(host, ttc::g_tl, bytes);
}
extern "C" int ttc_timeline_units_read(void* host, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(host, ttc::g_tlu, bytes);
}
extern "C" int ttc_timeline_bwd_warps_read(void* host, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(host, ttc::g_tlk, bytes);
}
static cudaStream_t g_probe_stream = 0;
extern "C" void ttc_probe_set_stream(void* st) { g_probe_stream = static_cast<cudaStream_t>(st); }
// An empty kernel of the same parameter size as the engine, and one with none.
__global__ void probe_big_param(const __grid_constant__ ttc::EngProgram p) {
  if (threadIdx.x == 0 && p.ntasks == 12345) ttc::g_status.code = 1;
}
__global__ void probe_small_param(int v) {
  if (threadIdx.x == 0 && v == 12345) ttc::g_status.code = 1;
}
extern "C" int ttc_probe_empty(int big, int coop, int grid, int threads, int smem) {
  ttc::EngProgram p;
  cudaFuncSetAttribute(probe_big_param, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  cudaFuncSetAttribute(probe_small_param, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (big)
    return (int)ttc::launch_ex(probe_big_param, dim3(grid), dim3(threads), smem, g_probe_stream, coop != 0, p);
  return (int)ttc::launch_ex(probe_small_param, dim3(grid), dim3(threads), smem, g_probe_stream, coop != 0, 0);
}
// Engine microbenchmark (timeline builds only): one program of `phases`
// phases, each holding `ntasks` GEMM tasks of m x n x k (f32, all operands
// in the given device buffer), or empty units when m == 0.
extern "C" int ttc_probe_engine(int phases, int ntasks, int units_if_empty, long m, long n, long k,
                                void* buf, int split) {
  using namespace ttc;
  EngBuilder b;
  float* f = static_cast<float*>(buf);
  for (int ph = 0; ph < phases; ++ph) {
    b.begin_phase();
    for (int t = 0; t < ntasks; ++t) {
      EngTask* task = b.add();
      if (m == 0) {
        task->kind = 99;
        task->units = units_if_empty;
        continue;
      }
      GemmArgs g;
      // split == 2: every phase reads its own operands (no reuse of cached lines)
      const size_t po = split == 2 ? (size_t)ph * (m * k + k * n + m * n) : 0;
      g.m = m; g.n = n; g.k = k;
      g.A = f + po; g.sam = k; g.sak = 1;
      g.B = f + po + m * k; g.sbk = n; g.sbn = 1;
      g.C = f + po + m * k + k * n + (size_t)t * m * n; g.scm = n; g.scn = 1;
      const bool sp = split == 1;
      eng_gemm_task(task, g, sp ? f + 4 * (m * k + k * n) + (size_t)t * m * n * 16 : nullptr,
                    sp ? (size_t)m * n * 16 : 0);
    }
  }
  b.end();
  // the barrier counter: one zeroed line past the operands
  b.p.bar = reinterpret_cast<unsigned long long*>(f + 8 * (m * k + k * n + m * n) + 64 * ntasks * m * n);
  cudaMemsetAsync(b.p.bar, 0, 256, g_probe_stream);
  return (int)eng_launch(b.p, g_probe_stream);
}

extern "C" int ttc_timeline_units_clear(void) {
  static unsigned long long zero[256 * 8 * 8];
  return (int)cudaMemcpyToSymbol(ttc::g_tlu, zero, sizeof(zero));
}
#endif
