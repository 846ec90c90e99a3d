// Tensor-core (tcgen05) path for bf16 activations: fused token-tile kernels.
#pragma once

#include "ttc_internal.h"

namespace ttc {

// Device addresses of the packed tensor-core operands and gradient sums.
struct TcPtrs {
  void* Anr = nullptr;   // bf16 [N][64]
  void* Bm = nullptr;    // bf16 [64][M]
  float* Dc = nullptr;   // [64] compacted middle diagonal (0 past r')
  int* rinfo = nullptr;  // [0] = r', [1 + c] = original index of column c
  float* dAc = nullptr;  // [N][64] sum over tokens of x^T dz
  float* dBc = nullptr;  // [M][64] sum over tokens of dy^T z'
  float* dDc = nullptr;  // [64]    sum over tokens of z * dz'
};
TcPtrs tc_ptrs(const LayerPlan& L, void* ws, size_t ws_off);

// True when the bf16 fused kernels handle this layer shape.
bool tc_supported(const LayerPlan& L);

// True when the E4M3-activation variants handle it too (row strides of x and
// dy in bytes must be multiples of 16 for TMA).
bool tc_f8_supported(const LayerPlan& L);

// Bytes of workspace the fused path needs for its packed operands.
size_t tc_operand_bytes(const LayerPlan& L);

// y = ((x A) diag(D_d)) B for T tokens; the packed operands (written by the
// merge engine's pack phase) are in the workspace at ws_off.  x is bf16, or
// E4M3 codes when f8; y is bf16.  With zs (256-byte aligned, T x 64 bf16) the
// kernel also stores z' = (x A) diag(D_d) there, rank compacted and padded.
// prefetch_x: the launch right before this one on the stream is the merge of
// the same call, which does not write x; the kernel then requests its first
// x boxes before waiting for that grid.
tt_status tc_forward(const LayerPlan& L, int64_t T, const void* x, void* y, void* ws,
                     size_t ws_off, bool f8, void* zs, bool prefetch_x, cudaStream_t st);

// Ranges of floats a backward token kernel sets to zero on its way: scratch
// that the merge backward then adds into, and the gradients that its
// one-phase program adds into.  Also zeroed when there are no tokens.
constexpr int kMaxZero = 6;
struct ZeroList {
  float* p[kMaxZero] = {};
  int n[kMaxZero] = {};
  int count = 0;
  // false when the list is full or the range is 2^31 floats or more
  bool add(float* ptr, size_t len) {
    if (!len) return true;
    if (count >= kMaxZero || len > 0x7FFFFFFF) return false;
    p[count] = ptr;
    n[count++] = (int)len;
    return true;
  }
};
// cudaMemsetAsync of every range (the no-token case)
cudaError_t zero_list_memset(const ZeroList& z, cudaStream_t st);

// dx for T tokens and the token sums dAc, dBc, dDc (zeroed by the pack
// phase, or, with det, written in a fixed order from per-CTA slots by one
// more kernel); the merge engine's unpack phase turns these into dA, dB, dD_d.
// The ranges of `zero` are set to 0 on the way, also when T == 0.  x and dy are bf16, or E4M3 codes when
// f8; dx is bf16.  With zs, z' is read from the forward's copy there instead
// of being recomputed from x.
// TT_DETERMINISTIC: per-CTA slots of the token sums (count CTAs at most):
// a [count][N][64], b [count][M][64], d [count][4][64] floats.
struct DetSlots {
  float* a = nullptr;
  float* b = nullptr;
  float* d = nullptr;
  int count = 0;
};
constexpr int kDetMaxSlots = 160;

tt_status tc_backward(const LayerPlan& L, int64_t T, const void* x, const void* dy, void* dx,
                      void* ws, size_t ws_off, const ZeroList& zero, bool f8,
                      const void* zs, const DetSlots* det, cudaStream_t st);

// ---- single-launch f32 path for small layers (small_f32.cu) -----------------
// True when one CTA's shared memory holds the whole pass for T tokens (f32
// activations, T <= 4096).
bool small_f32_supported(const LayerPlan& L, int64_t T);
// y = x W^T in one launch.  pout[k] (k < 2d, null entries skipped, pout itself
// may be null) receives the prefix product ending at core k, for a backward
// that reuses this forward's merge.
tt_status small_f32_forward(const LayerPlan& L, int64_t T, const void* x, const float* params,
                            void* y, float* const* pout, cudaStream_t st);
// dx and dparams (overwritten, or added to when acc) in one launch.
tt_status small_f32_backward(const LayerPlan& L, int64_t T, const void* x, const void* dy,
                             const float* params, void* dx, float* dparams, bool acc,
                             cudaStream_t st);

// ---- fused FFN pair (ffn_fused.cuh) -------------------------------------------
// True when both layers run on the tensor-core kernels and up's output width
// is down's input width.
bool ffn_tc_supported(const LayerPlan& U, const LayerPlan& D);

// y = TT_down(GELU(TT_up(x))) for T tokens, x and y bf16, with the hidden
// activations kept on the SM; each layer's packed operands are in the
// workspace at off1 / off2.  With zs1 and zs2 (T x 64 bf16 each) z1' and z2'
// are kept there for the backward.  y may be null when zs1 and zs2 are given:
// then only z1' and z2' are computed.
tt_status ffn_tc_forward(const LayerPlan& U, const LayerPlan& D, int64_t T, const void* x, void* y,
                         void* ws, size_t off1, size_t off2, void* zs1, void* zs2,
                         bool prefetch_x, cudaStream_t st);

// dx and both layers' token sums (dAc, dBc, dDc, zeroed beforehand) for T
// tokens from x, dy and the forward's z1', z2' (zs1, zs2); h, GELU(h), da and
// dh are recomputed per hidden chunk on the SM.  The ranges of `zero`
// are set to 0 on the way (the merge backward's scratch), also when T == 0.
// With det1 and det2 (TT_DETERMINISTIC, the up and down layer's slots) the
// token sums go through per-CTA slots summed in CTA order instead.
tt_status ffn_tc_backward(const LayerPlan& U, const LayerPlan& D, int64_t T, const void* x,
                          const void* dy, void* dx, void* ws, size_t off1, size_t off2,
                          const void* zs1, const void* zs2, const ZeroList& zero,
                          const DetSlots* det1, const DetSlots* det2, cudaStream_t st);

// The fixed-order sums of one layer's token-sum slots, filled by the `grid`
// CTAs of a deterministic token pass, into its dAc, dBc and dDc.
cudaError_t det_sum_launch(const LayerPlan& L, const DetSlots& det, int grid, float* dAc,
                           float* dBc, float* dDc, cudaStream_t st);

// ---- several layers on one input (qkv_fused.cuh) ----------------------------
// True when G (1..3) layers of equal input width all fit the tensor-core kernels.
bool multi_tc_supported(const LayerPlan* Ls, int G);

// y[g] = x W_g^T for every layer g, x streamed once; layer g's packed
// operands at offs[g] of ws.  With zs (G pointers, T x 64 bf16 each) every
// z'_g is kept there; y may be null when zs is given (then only z'_g).
tt_status multi_tc_forward(const LayerPlan* Ls, int G, int64_t T, const void* x, void* const* y,
                           void* ws, const size_t* offs, void* const* zs, bool prefetch_x,
                           cudaStream_t st);

// dx = sum_g dy[g] W_g and every layer's token sums (dAc, dBc, dDc, zeroed
// beforehand) from x, dy[g] and the forward's z'_g; x streamed once.
// The ranges of `zero` are set to 0 on the way, also when T == 0.  With det
// (TT_DETERMINISTIC, one DetSlots a layer) the token sums go through per-CTA
// slots summed in CTA order instead.
tt_status multi_tc_backward(const LayerPlan* Ls, int G, int64_t T, const void* x,
                            const void* const* dy, void* dx, void* ws, const size_t* offs,
                            const void* const* zs, const ZeroList& zero, const DetSlots* det,
                            cudaStream_t st);

}  // namespace ttc
