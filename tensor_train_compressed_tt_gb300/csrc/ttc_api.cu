// libttc C ABI: plans, parameter/workspace layout, argument checks and the
// orchestration of the kernels for one TT layer and for the GELU FFN pair.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "merge_engine.h"
#include "rank_step.cuh"
#include "tc_fused.h"
#include "ttc_internal.h"

namespace ttc {
namespace {

constexpr int64_t kMaxDim = 1 << 20;   // N, M
constexpr int kMaxRank = 4096;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

tt_status build_layer(const tt_desc* desc, LayerPlan* L) {
  if (!desc || !L) return TT_ERR_INVALID_ARG;
  const int d = desc->d;
  if (d < 1 || d > TT_MAX_D) return TT_ERR_INVALID_ARG;
  if (desc->act != TT_DT_F32 && desc->act != TT_DT_BF16 && desc->act != TT_DT_E4M3)
    return TT_ERR_INVALID_ARG;
  if (desc->flags & ~(TT_ACCUMULATE | TT_REUSE_MERGE | TT_REUSE_Z | TT_DETERMINISTIC))
    return TT_ERR_INVALID_ARG;
  LayerPlan p;
  p.d = d;
  p.K = 2 * d;
  p.act = desc->act;
  p.flags = desc->flags;
  if (p.flags & TT_REUSE_Z) p.flags |= TT_REUSE_MERGE;  // the kept z' implies the kept merge
  p.N = 1;
  p.M = 1;
  for (int k = 0; k < d; ++k) {
    if (desc->in_modes[k] < 1 || desc->out_modes[k] < 1) return TT_ERR_INVALID_ARG;
    p.s[k] = desc->in_modes[k];
    p.s[d + k] = desc->out_modes[k];
    p.N *= desc->in_modes[k];
    p.M *= desc->out_modes[k];
    if (p.N > kMaxDim || p.M > kMaxDim) return TT_ERR_UNSUPPORTED;
  }
  for (int k = 0; k <= p.K; ++k) {
    p.r[k] = desc->ranks[k];
    if (p.r[k] < 1 || p.r[k] > kMaxRank) return TT_ERR_INVALID_ARG;
  }
  if (p.r[0] != 1 || p.r[p.K] != 1) return TT_ERR_INVALID_ARG;
  p.rd = p.r[d];
  size_t off = 0;
  for (int k = 0; k < p.K; ++k) {
    p.core_off[k] = off;
    off += (size_t)p.r[k] * p.s[k] * p.r[k + 1];
  }
  for (int e = 0; e < p.K - 1; ++e) {
    p.diag_off[e] = off;
    off += (size_t)p.r[e + 1];
  }
  p.n_floats = off;
  // rows of the merged prefix ending at core k
  int64_t u = 1;
  for (int k = 0; k < d; ++k) {
    u *= p.s[k];
    p.U[k] = u;
  }
  u = p.rd;
  for (int k = d; k < p.K; ++k) {
    u *= p.s[k];
    p.U[k] = u;
  }
  // the merge kernels index every matrix they touch in 32 bits: the packed
  // parameters, each prefix product (U_k x r_{k+1}, A and B among them)
  constexpr int64_t kMax32 = (int64_t)1 << 31;
  if ((int64_t)p.n_floats >= kMax32) return TT_ERR_UNSUPPORTED;
  for (int k = 0; k < p.K; ++k)
    if (p.U[k] * p.r[k + 1] >= kMax32) return TT_ERR_UNSUPPORTED;
  *L = p;
  return TT_OK;
}

// ---- workspace ------------------------------------------------------------
struct WsLayout {
  size_t P[kMaxK] = {};  // merged chain prefixes (floats), 0 where aliased to params
  size_t dA = 0, dB = 0;
  size_t bar = 0;        // grid-barrier counter of the merge programs (one 256-byte line,
                         // directly before q: the backward token pass zeroes both at once)
  size_t q = 0;          // reverse-chain dQ buffers: step j of side s at q + (2j + s) * qstride
  size_t qstride = 0;    // floats between dQ buffers
  size_t part[4] = {};   // split-K partials (input side 0/1, output 2/3)
  size_t part_cap = 0;   // floats per partial buffer
  size_t z = 0, dzp = 0; // SIMT token path intermediates
  size_t tc = 0;         // tensor-core path operands
  size_t zs = 0;         // z' kept by the forward for the backward (TT_REUSE_Z), bf16 [T][64]
  size_t det = 0;        // TT_DETERMINISTIC: per-CTA token-sum slots (det_slots of them)
  int det_slots = 0;
  size_t end = 0;        // end of this layer's scratch
};

size_t chain_len(const LayerPlan& L, int k) { return (size_t)L.U[k] * L.r[k + 1]; }

size_t layer_layout(const LayerPlan& L, int64_t T, size_t base, WsLayout* w,
                    bool simt_tokens = false, bool keep_z = false) {
  size_t off = align_up(base, 256);
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  size_t qmax = 0, pmax = 0;
  for (int k = 0; k < L.K; ++k) {
    size_t n = chain_len(L, k);
    if (n > qmax) qmax = n;
    size_t pf = eng_partial_floats(L.r[k], (int64_t)L.s[k] * L.r[k + 1], 0);
    if (pf > pmax) pmax = pf;
    w->P[k] = (k == 0 || k == L.d) ? 0 : take(n * sizeof(float));
  }
  w->dA = take((size_t)L.N * L.rd * sizeof(float));
  w->dB = take((size_t)L.rd * L.M * sizeof(float));
  w->qstride = align_up(qmax * sizeof(float), 256) / sizeof(float);
  w->bar = take(256);
  w->q = take(2 * (TT_MAX_D - 1) * w->qstride * sizeof(float));
  for (int i = 0; i < 4; ++i) w->part[i] = take(pmax * sizeof(float));
  w->part_cap = pmax;
  const bool tc = !simt_tokens && tc_supported(L) && L.act != TT_DT_F32;
  w->z = take(tc ? 0 : (size_t)T * L.rd * sizeof(float));
  w->dzp = take(tc ? 0 : (size_t)T * L.rd * sizeof(float));
  w->tc = take(tc_operand_bytes(L));
  w->zs = take(tc && (keep_z || (L.flags & TT_REUSE_Z)) ? (size_t)T * 64 * 2 : 0);
  // one slot per CTA of the backward token pass (128-token tiles, at most
  // kDetMaxSlots CTAs): [N + M + 4][64] floats each
  w->det_slots = 0;
  if (tc && (L.flags & TT_DETERMINISTIC)) {
    const int64_t tiles = (T + 127) / 128;
    w->det_slots = (int)(tiles < kDetMaxSlots ? (tiles > 0 ? tiles : 1) : kDetMaxSlots);
  }
  w->det = take((size_t)w->det_slots * (size_t)(L.N + L.M + 4) * 64 * sizeof(float));
  w->end = off;
  return off;
}

// The TT_DETERMINISTIC token-sum slots of a layer's workspace region:
// det_slots x [N][64] for dA, then x [M][64] for dB, then x [4][64] for dD.
DetSlots det_slots(const LayerPlan& L, void* ws, const WsLayout& w) {
  DetSlots d;
  if (w.det_slots) {
    d.count = w.det_slots;
    d.a = reinterpret_cast<float*>(static_cast<char*>(ws) + w.det);
    d.b = d.a + (size_t)w.det_slots * L.N * 64;
    d.d = d.b + (size_t)w.det_slots * L.M * 64;
  }
  return d;
}

struct FfnLayout {
  WsLayout up, down;
  size_t h = 0, a = 0, da = 0, end = 0;
};

// Both layers of a bf16 FFN pair run on the tensor-core path with bf16
// intermediates h, a = GELU(h), da; otherwise on the SIMT path in f32.
bool ffn_tc(const tt_plan_s* p) {
  return p->L[0].act == TT_DT_BF16 && tc_supported(p->L[0]) && tc_supported(p->L[1]);
}

// A bf16 FFN pair whose layers both fit the tensor-core kernels runs fused:
// h, GELU(h), da and dh never leave the SM (under TT_DETERMINISTIC too, the
// token sums then going through per-CTA slots).  TTC_FFN_UNFUSED=1 selects
// the layer-by-layer path instead (a measurement aid).
bool ffn_fused(const tt_plan_s* p) {
  static int off = -1;
  if (off < 0) {
    const char* e = getenv("TTC_FFN_UNFUSED");
    off = (e && e[0] && e[0] != '0') ? 1 : 0;
  }
  return !off && ffn_tc(p) && ffn_tc_supported(p->L[0], p->L[1]);
}

// Without the reuse flags the two layers' scratch shares one region; with
// them each layer keeps its merges (and z') from the forward in a region of
// its own.
size_t ffn_layout(const tt_plan_s* p, int64_t T, FfnLayout* f) {
  if (ffn_fused(p)) {
    // both layers' operands at once, and their z' (T x 64 bf16 each), which
    // the backward reads: no T x hidden buffers
    size_t e0 = layer_layout(p->L[0], T, 256, &f->up, false, true);
    size_t e1 = layer_layout(p->L[1], T, align_up(e0, 256), &f->down, false, true);
    f->h = f->a = f->da = 0;
    f->end = align_up(e1, 256);
    return f->end;
  }
  const bool tc = ffn_tc(p);
  const bool keep = (p->L[0].flags & TT_REUSE_MERGE) != 0;
  size_t e0 = layer_layout(p->L[0], T, 256, &f->up, !tc);
  size_t e1 = layer_layout(p->L[1], T, keep ? align_up(e0, 256) : 256, &f->down, !tc);
  size_t off = align_up(e0 > e1 ? e0 : e1, 256);
  const size_t hb = (size_t)T * p->L[0].M * (tc ? 2 : sizeof(float));
  f->h = off;
  off = align_up(off + hb, 256);
  f->a = off;
  off = align_up(off + hb, 256);
  f->da = off;
  off = align_up(off + hb, 256);
  f->end = off;
  return off;
}

#define TT_CUDA(call)                                      \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return TT_ERR_CUDA;             \
  } while (0)

float* fptr(void* ws, size_t off) { return reinterpret_cast<float*>(static_cast<char*>(ws) + off); }

// Chain prefix pointers: P_k = reshape((P_{k-1} * D_{k-1}) . G_k) on each side;
// P_0 and P_d are the first cores themselves.
void chain_ptrs(const LayerPlan& L, const float* params, void* ws, const WsLayout& w,
                const float** P) {
  for (int k = 0; k < L.K; ++k)
    P[k] = (k == 0 || k == L.d) ? params + L.core_off[k] : fptr(ws, w.P[k]);
}

// ---- merge programs ---------------------------------------------------------
// out[0 .. n) = 0 as one engine task.
void eng_zero_task(EngBuilder& b, float* out, int64_t n) {
  EngTask* z = b.add();
  z->kind = kEScale;
  z->n = n;
  z->chunk = 8192;  // a unit's cost is mostly fixed: few large units keep a phase in one wave
  z->units = (int)((n + z->chunk - 1) / z->chunk);
  z->x = nullptr;
  z->out = out;
  z->acc = 0;
}

// dQ scratch of reverse step j on side s (0 input, 1 output).
float* dq_buf(void* ws, const WsLayout& w, int j, int side) {
  return fptr(ws, w.q) + (size_t)(2 * j + side) * w.qstride;
}


// Forward merge: phase j computes P_j (input side) and P_{d+j} (output side).
// On the tensor-core path the GEMMs that produce A and B also write the
// compacted bf16 operands, and the first phase writes the padding and the
// metadata (and zeroes the token sums for a backward call).
// Fallback for chains with an internal rank above 64: one GEMM phase per
// chain step (grid barriers in between).
tt_status run_merge_forward_gemm(const LayerPlan& L, const float* params, void* ws, const WsLayout& w,
                            const float** P, bool pack, bool zero_grads, cudaStream_t st) {
  chain_ptrs(L, params, ws, w, P);
  const float* Dmid = params + L.diag_off[L.d - 1];
  const TcPtrs tc = pack ? tc_ptrs(L, ws, w.tc) : TcPtrs();
  EngBuilder b;
  if (L.d == 1 && pack) {
    b.begin_phase();
    eng_pack_task(b.add(), L, P[0], P[1], Dmid, tc, zero_grads, false);
  }
  for (int j = 1; j < L.d; ++j) {
    b.begin_phase();
    if (pack && j == 1) eng_pack_task(b.add(), L, nullptr, nullptr, Dmid, tc, zero_grads, true);
    for (int k : {j, L.d + j}) {
      GemmArgs g;
      g.m = L.U[k - 1];
      g.n = (int64_t)L.s[k] * L.r[k + 1];
      g.k = L.r[k];
      g.A = P[k - 1]; g.sam = L.r[k]; g.sak = 1;
      g.kscale = params + L.diag_off[k - 1]; g.klen = L.r[k];
      g.B = params + L.core_off[k]; g.sbk = g.n; g.sbn = 1;
      g.C = const_cast<float*>(P[k]); g.scm = g.n; g.scn = 1;
      EngTask* t = b.add();
      eng_gemm_task(t, g, nullptr, 0);
      if (pack && j == L.d - 1) {
        t->pack_side = (k == j) ? 1 : 2;
        t->tc = tc;
        t->s = Dmid;
        t->rd = L.rd;
        t->N = (int)L.N;
        t->M = (int)L.M;
      }
    }
  }
  b.end();
  if (b.overflow) return TT_ERR_UNSUPPORTED;
  if (b.p.nphases == 0) return TT_OK;
  b.p.bar = reinterpret_cast<unsigned long long*>(fptr(ws, w.bar));
  if (b.p.nphases > 1) TT_CUDA(cudaMemsetAsync(b.p.bar, 0, 256, st));
  TT_CUDA(eng_launch(b.p, st));
  return TT_OK;
}

// The one-phase chain program of one layer's forward merge, added to the
// builder's current phase; false when a chain does not fit the chain units
// (ranks above 64 or cores too large to stage): then the GEMM-phase program
// below serves.
bool add_merge_forward(EngBuilder& b, const LayerPlan& L, const float* params, void* ws,
                       const WsLayout& w, const float** P, bool pack, bool zero_grads) {
  chain_ptrs(L, params, ws, w, P);
  const float* Dmid = params + L.diag_off[L.d - 1];
  const TcPtrs tc = pack ? tc_ptrs(L, ws, w.tc) : TcPtrs();
  if (L.d == 1) {
    if (pack) eng_pack_task(b.add(), L, P[0], P[1], Dmid, tc, zero_grads, false);
  } else {
    // one phase: each side's rows recomputed per prefix (no grid barrier);
    // padding, metadata and the zeroed token sums come from the pack task
    if (pack) eng_pack_task(b.add(), L, nullptr, nullptr, Dmid, tc, zero_grads, true);
    for (int side = 0; side < 2; ++side) {
      const int k0 = side == 0 ? 0 : L.d;
      ChainDesc c;
      c.L = L.d;
      c.r[0] = L.r[k0];
      int64_t np = side == 0 ? 1 : L.rd;
      for (int k = 0; k < L.d; ++k) {
        c.core[k] = params + L.core_off[k0 + k];
        c.s[k] = L.s[k0 + k];
        c.r[k + 1] = L.r[k0 + k + 1];
        if (k < L.d - 1) {
          c.diag[k] = params + L.diag_off[k0 + k];
          np *= L.s[k0 + k];
        }
        if (k >= 1 && k <= L.d - 2) c.prow[k] = const_cast<float*>(P[k0 + k]);
      }
      // the f32 A / B are read only by the SIMT token path; the tensor-core
      // path takes the packed bf16 operands alone
      c.out = pack ? nullptr : const_cast<float*>(P[k0 + L.d - 1]);
      c.nprefix = np;
      EngTask t;
      if (!eng_chain_task(&t, c)) return false;  // ranks above 64 or cores too large to stage
      if (pack) {
        t.pack_side = side + 1;
        t.tc = tc;
        t.s = Dmid;
        t.rd = L.rd;
        t.N = (int)L.N;
        t.M = (int)L.M;
      }
      *b.add() = t;
    }
  }
  return true;
}

bool chain_merge_fits(const LayerPlan& L, const float* params, void* ws, const WsLayout& w) {
  EngBuilder probe;
  probe.begin_phase();
  const float* P[kMaxK];
  return add_merge_forward(probe, L, params, ws, w, P, false, false) && !probe.overflow;
}

tt_status run_merge_forward(const LayerPlan& L, const float* params, void* ws, const WsLayout& w,
                            const float** P, bool pack, bool zero_grads, cudaStream_t st) {
  if (!chain_merge_fits(L, params, ws, w))
    return run_merge_forward_gemm(L, params, ws, w, P, pack, zero_grads, st);
  EngBuilder b;
  b.begin_phase();
  add_merge_forward(b, L, params, ws, w, P, pack, zero_grads);
  b.end();
  if (b.overflow) return TT_ERR_UNSUPPORTED;
  if (b.p.ntasks == 0) return TT_OK;
  TT_CUDA(eng_launch(b.p, st));
  return TT_OK;
}

// The forward merges of n layers in one launch where they all fit the chain
// units and the program's task table (else one launch each).
tt_status run_merge_forward_n(int n, const LayerPlan* const* Ls, const float* const* params,
                              const WsLayout* const* wl, const float** const* P, void* ws,
                              bool zero_grads, cudaStream_t st) {
  bool fit = true;
  for (int i = 0; i < n && fit; ++i) fit = chain_merge_fits(*Ls[i], params[i], ws, *wl[i]);
  if (fit) {
    EngBuilder b;
    b.begin_phase();
    for (int i = 0; i < n; ++i) add_merge_forward(b, *Ls[i], params[i], ws, *wl[i], P[i], true, zero_grads);
    b.end();
    if (!b.overflow) {
      if (b.p.ntasks > 0) TT_CUDA(eng_launch(b.p, st));
      return TT_OK;
    }
  }
  for (int i = 0; i < n; ++i) {
    tt_status s = run_merge_forward(*Ls[i], params[i], ws, *wl[i], P[i], true, zero_grads, st);
    if (s != TT_OK) return s;
  }
  return TT_OK;
}

// Both layers' forward merges of an FFN pair.
tt_status run_merge_forward2(const LayerPlan& U, const float* pu, const WsLayout& wu,
                             const float** PU, const LayerPlan& D, const float* pd,
                             const WsLayout& wd, const float** PD, void* ws, bool zero_grads,
                             cudaStream_t st) {
  const LayerPlan* Ls[2] = {&U, &D};
  const float* params[2] = {pu, pd};
  const WsLayout* wl[2] = {&wu, &wd};
  const float** P[2] = {PU, PD};
  return run_merge_forward_n(2, Ls, params, wl, P, ws, zero_grads, st);
}

// Backward through the merges.  For one side with cores k_first..k_last and
// dP_{k_last} = dlast, reverse step k (k_last down to k_first+1) computes
//   dG_k = diag(D_{k-1}) P_{k-1}^T Y,  dQ = Y G_k^T,  dD_{k-1} = colsum(P_{k-1} * dQ)
// with Y = dlast for the first step and Y = dQ_prev * D_k afterwards; the
// first core gets dG = Y * D_{k_first}.  Both sides advance in lockstep, one
// phase per step; split-K partials of the first step's dG are reduced in the
// next phase.  With two or more steps a side, the last step's dQ GEMM writes
// the first core's dG and dD straight from its epilogue (no phase of its
// own), the later steps' dG add their K splits atomically, and every dQ is
// added atomically into zeroed scratch: step 0's by the backward token pass
// (dq0_zero_floats), the others' by phase 0, which also zeroes the gradient
// slices that later phases add into (unless accumulating).
size_t dq0_zero_floats(const LayerPlan& L, const WsLayout& w) {
  return L.d >= 3 ? 2 * (size_t)(L.d - 2) * w.qstride : 0;  // steps 0 .. d-3, both sides
}

// The backward merge folds its last reverse step into the first core's
// gradient (atomics), for order 6 and up without TT_DETERMINISTIC.
bool merge_fold(const LayerPlan& L) { return L.d >= 3 && !(L.flags & TT_DETERMINISTIC); }

// What the backward token pass zeroes on its way: the merge program's
// grid-barrier line and the step-0 dQ scratch right after it.
float* bwd_zero_ptr(void* ws, const WsLayout& w) { return fptr(ws, w.bar); }
size_t bwd_zero_floats(const LayerPlan& L, const WsLayout& w) {
  return (w.q - w.bar) / sizeof(float) + dq0_zero_floats(L, w);
}

// What the backward token pass zeroes on its way: the merge program's
// grid-barrier line and the dQ scratch right after it, and (folded merge,
// not accumulating) the whole of dparams, whose parts the merge's later
// phases add into.
bool bwd_zero_add(ZeroList* z, const LayerPlan& L, void* ws, const WsLayout& w, float* dparams,
                  bool acc) {
  if (!z->add(bwd_zero_ptr(ws, w), bwd_zero_floats(L, w))) return false;
  return acc || !merge_fold(L) || z->add(dparams, L.n_floats);
}

// The merge-backward program of one layer, built phase by phase so that the
// programs of several layers (the two of an FFN pair) can share one launch.
struct MergeBwd {
  const LayerPlan& L;
  const float* params;
  const float** P;
  float* dparams;
  bool acc, unpack, rezero;
  void* ws;
  const WsLayout& w;
  int steps = 0, pre = 0, nphases = 0;
  bool fold = false;
  TcPtrs tc;
  // the rank-adaptive step as one more phase, after every read of params
  const RankStep* rank = nullptr;
  float* params_mut = nullptr;
  struct Side {
    int k_first, k_last;
    const float* Y;
    const float* yscale;
    int qs, pi;          // side index of the dQ buffers, base index of part buffers
    int flip;
    int pending;         // task index of a split GEMM whose partials the next phase reduces
    const float* dQ;     // last dQ (for coldot in the next phase)
    int coldot_k;        // link whose dD the next phase computes (-1: none)
  } sides[2];

  MergeBwd(const LayerPlan& L_, const float* params_, const float** P_, const float* dA,
           const float* dB, float* dparams_, bool acc_, bool unpack_, bool rezero_, void* ws_,
           const WsLayout& w_)
      : L(L_), params(params_), P(P_), dparams(dparams_), acc(acc_), unpack(unpack_),
        rezero(rezero_), ws(ws_), w(w_) {
    steps = L.d - 1;
    tc = unpack ? tc_ptrs(L, ws, w.tc) : TcPtrs();
    // order 2: the merges are the cores themselves; unpack in full first
    pre = (unpack && steps == 0) ? 1 : 0;
    // the folded last step adds into the first core's gradient with atomics;
    // TT_DETERMINISTIC takes the unfolded program (split partials reduced in
    // split order, dD by column sums)
    fold = merge_fold(L);
    nphases = pre + (fold ? steps : steps + 1);
    sides[0] = {0, L.d - 1, dA, nullptr, 0, 0, 0, -1, nullptr, -1};
    sides[1] = {L.d, L.K - 1, dB, nullptr, 1, 2, 0, -1, nullptr, -1};
  }

  // The tasks of phase jj (the builder's current phase).
  void add_phase(EngBuilder& b, int jj) {
    if (jj < pre) {
      eng_unpack_task(b.add(), L, tc, params + L.diag_off[L.d - 1], fptr(ws, w.dA),
                      fptr(ws, w.dB), dparams + L.diag_off[L.d - 1], acc);
      return;
    }
    const int j = jj - pre;
    const int last_phase = nphases - pre - 1;
    const int mode = acc ? kAccumulate : kStore;
    if (unpack && steps > 0 && j == 0)
      eng_dd_task(b.add(), L, tc, params + L.diag_off[L.d - 1], dparams + L.diag_off[L.d - 1],
                  acc);
    // (folded: the dQ scratch and, unless accumulating, dparams were zeroed
    // by the backward token pass, see bwd_zero_add)
    for (Side& sd : sides) {
      // work left over from the previous step
      if (sd.pending >= 0) {  // the previous phase is balanced by now
        const EngTask prev = b.p.t[sd.pending];
        if (prev.splits > 1 && prev.partial) eng_gemm_final_task(b.add(), prev);
        sd.pending = -1;
      }
      if (sd.coldot_k >= 0) {
        const int k = sd.coldot_k;  // dD_{k-1} from P_{k-1} and dQ_k
        EngTask* t = b.add();
        t->kind = kEColdot;
        t->units = L.r[k];
        t->x = P[k - 1]; t->sx = L.r[k];
        t->y = sd.dQ; t->sy = L.r[k];
        t->n = L.U[k - 1];
        t->s = params + L.diag_off[k - 1];
        t->out = dparams + L.diag_off[k - 1];
        t->acc = acc ? 1 : 0;
        sd.coldot_k = -1;
      }
      if (j < steps) {
        const int k = sd.k_last - j;
        const int rk = L.r[k], rk1 = L.r[k + 1];
        const int64_t U = L.U[k - 1];
        const int64_t ncol = (int64_t)L.s[k] * rk1;
        const bool last = j == steps - 1;
        const int gat = (unpack && j == 0) ? (&sd == &sides[0] ? 1 : 2) : 0;
        GemmArgs g;  // dG_k
        g.m = rk; g.n = ncol; g.k = U;
        g.A = P[k - 1]; g.sam = 1; g.sak = rk;
        g.B = sd.Y; g.sbk = ncol; g.sbn = 1;
        g.rscale = params + L.diag_off[k - 1];
        g.cscale = sd.yscale; g.clen = rk1;
        g.C = dparams + L.core_off[k]; g.scm = ncol; g.scn = 1;
        EngTask* t = b.add();
        if (fold && j >= 1) {  // added into zeroed (or accumulated) dparams
          g.mode = kAtomic;
          eng_gemm_task(t, g, nullptr, 0, true);
        } else {
          g.mode = mode;
          eng_gemm_task(t, g, fptr(ws, w.part[sd.pi + (sd.flip & 1)]), w.part_cap);
        }
        if (gat) {  // read dA / dB straight from the compacted token sums
          t->gather = gat;
          t->gather_op = 1;
          t->s = params + L.diag_off[L.d - 1];
          t->tc = tc;
          t->rd = L.rd;
          t->M = (int)L.M;
        }
        if (!b.overflow && t->partial) sd.pending = (int)(t - b.p.t);
        GemmArgs h;  // dQ = Y G_k^T
        h.m = U; h.n = rk; h.k = ncol;
        h.A = sd.Y; h.sam = ncol; h.sak = 1;
        h.kscale = sd.yscale; h.klen = rk1;
        h.B = params + L.core_off[k]; h.sbk = 1; h.sbn = ncol;
        h.scm = rk; h.scn = 1;
        EngTask* th = b.add();
        float* dQ = nullptr;
        if (fold && last) {
          // the first core: dG = dQ * D_{k_first}, dD_{k_first} = colsum(P_{k_first} * dQ)
          const int kf = sd.k_first;
          h.mode = kAtomic;
          h.cscale = params + L.diag_off[kf]; h.clen = rk;
          eng_gemm_task(th, h, nullptr, 0, true);
          th->fold_g = dparams + L.core_off[kf];
          th->fold_p = P[kf];
          th->fold_dd = dparams + L.diag_off[kf];
        } else {
          dQ = dq_buf(ws, w, j, sd.qs);
          h.C = dQ;
          h.mode = fold ? kAtomic : kStore;
          eng_gemm_task(th, h, nullptr, 0, fold);
        }
        if (gat) {
          th->gather = gat;
          th->gather_op = 0;
          th->s = params + L.diag_off[L.d - 1];
          th->tc = tc;
          th->rd = L.rd;
          th->M = (int)L.M;
        }
        sd.dQ = dQ;
        sd.coldot_k = (fold && last) ? -1 : k;
        sd.Y = dQ;
        sd.yscale = params + L.diag_off[k - 1];
        sd.flip ^= 1;
      } else {
        // (only without folding) first core of the side
        EngTask* t = b.add();
        t->kind = kEScale;
        t->n = (int64_t)L.r[sd.k_first] * L.s[sd.k_first] * L.r[sd.k_first + 1];
        t->units = (int)((t->n + 1023) / 1024);
        t->x = sd.Y;
        t->s = sd.yscale;
        t->len = L.r[sd.k_first + 1];
        t->out = dparams + L.core_off[sd.k_first];
        t->acc = acc ? 1 : 0;
      }
    }
    if (rezero && j == last_phase && (j >= 1 || steps == 0)) {
      // leave the token sums zeroed for the next backward that reuses this
      // workspace's merge (read only by an earlier phase: the first reverse
      // step, or the unpack phase for order 2); dAc, dBc and dDc are adjacent
      eng_zero_task(b, const_cast<float*>(tc.dAc), (L.N + L.M + 1) * 64);
    }
  }
};

tt_status run_merge_backward_multi(MergeBwd* const* layers, int n, cudaStream_t st) {
  EngBuilder b;
  const int nph = layers[0]->nphases;
  for (int i = 1; i < n; ++i)
    if (layers[i]->nphases != nph || layers[i]->pre != layers[0]->pre) return TT_ERR_UNSUPPORTED;
  for (int j = 0; j < nph; ++j) {
    b.begin_phase();
    for (int i = 0; i < n; ++i) layers[i]->add_phase(b, j);
  }
  bool any_rank = false;
  for (int i = 0; i < n; ++i) any_rank |= layers[i]->rank != nullptr;
  if (any_rank) {
    b.begin_phase();
    for (int i = 0; i < n; ++i)
      if (layers[i]->rank)
        eng_rank_task(b.add(), layers[i]->L, layers[i]->params_mut, layers[i]->dparams,
                      *layers[i]->rank);
  }
  b.end();
  if (b.overflow) return TT_ERR_UNSUPPORTED;
  if (b.p.nphases == 0) return TT_OK;
  // one barrier line serves the program: the first layer's, zeroed by the
  // backward token pass that comes before in the stream
  b.p.bar = reinterpret_cast<unsigned long long*>(fptr(layers[0]->ws, layers[0]->w.bar));
  TT_CUDA(eng_launch(b.p, st));
  return TT_OK;
}

tt_status run_merge_backward(const LayerPlan& L, const float* params, const float** P,
                             const float* dA, const float* dB, float* dparams, bool acc,
                             bool unpack, bool rezero, void* ws, const WsLayout& w,
                             cudaStream_t st, const RankStep* rank = nullptr,
                             float* params_mut = nullptr) {
  MergeBwd m(L, params, P, dA, dB, dparams, acc, unpack, rezero, ws, w);
  m.rank = rank;
  m.params_mut = params_mut;
  MergeBwd* one = &m;
  return run_merge_backward_multi(&one, 1, st);
}

// ---- one layer ---------------------------------------------------------------
// Output dtype of a layer: bf16 for E4M3 inputs, else the input dtype.
int out_dtype(int act) { return act == TT_DT_E4M3 ? TT_DT_BF16 : act; }

// The fused tensor-core kernels take bf16 or E4M3 inputs and write bf16.
bool use_tc(const LayerPlan& L, int tx, int ty) {
  if (tx == TT_DT_E4M3) return ty == TT_DT_BF16 && tc_f8_supported(L);
  return tx == TT_DT_BF16 && ty == TT_DT_BF16 && L.act == TT_DT_BF16 && tc_supported(L);
}

// Small f32 layers run as one launch per pass (merges, token products and
// gradients in one CTA's shared memory).
bool use_small(const LayerPlan& L, int64_t T, int tx, int ty) {
  return tx == TT_DT_F32 && ty == TT_DT_F32 && small_f32_supported(L, T);
}

tt_status layer_forward(const LayerPlan& L, int64_t T, const void* x, int tx, const float* params,
                        void* y, int ty, void* ws, const WsLayout& w, cudaStream_t st) {
  const float* P[kMaxK];
  if (use_small(L, T, tx, ty)) {
    // with TT_REUSE_MERGE the prefix products go where the merge engine
    // would have left them (the backward may take another path)
    float* pout[kMaxK] = {};
    if (L.flags & TT_REUSE_MERGE) {
      chain_ptrs(L, params, ws, w, P);
      for (int k = 0; k < L.K; ++k)
        if (k != 0 && k != L.d) pout[k] = const_cast<float*>(P[k]);
    }
    prof_begin(kPhFwd, st);
    tt_status s = small_f32_forward(L, T, x, params, y, pout, st);
    prof_end(kPhFwd, st);
    return s;
  }
  const bool tc = use_tc(L, tx, ty);
  if (!tc && tx == TT_DT_E4M3) return TT_ERR_UNSUPPORTED;  // E4M3 runs on the fused kernels only
  const bool reuse = (L.flags & TT_REUSE_MERGE) != 0;
  prof_begin(kPhMerge, st);
  tt_status s = run_merge_forward(L, params, ws, w, P, tc, reuse, st);
  prof_end(kPhMerge, st);
  if (s != TT_OK) return s;
  prof_begin(kPhFwd, st);
  if (tc) {
    void* zs = (L.flags & TT_REUSE_Z) ? static_cast<char*>(ws) + w.zs : nullptr;
    s = tc_forward(L, T, x, y, ws, w.tc, tx == TT_DT_E4M3, zs, true, st);  // after the merge
  } else {
    const float* A = P[L.d - 1];   // N x rd
    const float* B = P[L.K - 1];   // rd x M
    const float* Dm = params + L.diag_off[L.d - 1];
    float* z = fptr(ws, w.z);
    GemmArgs g;
    g.m = T; g.n = L.rd; g.k = L.N;
    g.A = x; g.sam = L.N; g.sak = 1; g.ta = tx;
    g.B = A; g.sbk = L.rd; g.sbn = 1;
    g.C = z; g.scm = L.rd; g.scn = 1;
    cudaError_t e = gemm_simt(g, st);
    if (e == cudaSuccess) {
      GemmArgs h;
      h.m = T; h.n = L.M; h.k = L.rd;
      h.A = z; h.sam = L.rd; h.sak = 1;
      h.kscale = Dm; h.klen = L.rd;
      h.B = B; h.sbk = L.M; h.sbn = 1;
      h.C = y; h.scm = L.M; h.scn = 1; h.tc = ty;
      e = gemm_simt(h, st);
    }
    s = e == cudaSuccess ? TT_OK : TT_ERR_CUDA;
  }
  prof_end(kPhFwd, st);
  return s;
}

// SIMT token pass of the backward: dx, dD_d, and dA / dB sums over tokens.
tt_status simt_backward_tokens(const LayerPlan& L, int64_t T, const void* x, int tx,
                               const void* dy, int tdy, const float* params, const float** P,
                               void* dx, int tdx, float* dparams, bool acc, void* ws,
                               const WsLayout& w, cudaStream_t st) {
  const float* A = P[L.d - 1];
  const float* B = P[L.K - 1];
  const float* Dm = params + L.diag_off[L.d - 1];
  float* dA = fptr(ws, w.dA);
  float* dB = fptr(ws, w.dB);
  TT_CUDA(cudaMemsetAsync(dA, 0, (size_t)L.N * L.rd * sizeof(float), st));
  TT_CUDA(cudaMemsetAsync(dB, 0, (size_t)L.rd * L.M * sizeof(float), st));
  if (T == 0) {
    if (!acc) TT_CUDA(cudaMemsetAsync(dparams + L.diag_off[L.d - 1], 0, L.rd * sizeof(float), st));
    return TT_OK;
  }
  float* z = fptr(ws, w.z);
  float* dzp = fptr(ws, w.dzp);
  GemmArgs g;  // z = x A
  g.m = T; g.n = L.rd; g.k = L.N;
  g.A = x; g.sam = L.N; g.sak = 1; g.ta = tx;
  g.B = A; g.sbk = L.rd; g.sbn = 1;
  g.C = z; g.scm = L.rd; g.scn = 1;
  TT_CUDA(gemm_simt(g, st));
  GemmArgs h;  // dz' = dy B^T
  h.m = T; h.n = L.rd; h.k = L.M;
  h.A = dy; h.sam = L.M; h.sak = 1; h.ta = tdy;
  h.B = B; h.sbk = 1; h.sbn = L.M;
  h.C = dzp; h.scm = L.rd; h.scn = 1;
  TT_CUDA(gemm_simt(h, st));
  // dD_d = sum_t z * dz'
  TT_CUDA(coldot(T, L.rd, z, L.rd, dzp, L.rd, Dm, dparams + L.diag_off[L.d - 1], acc, st));
  GemmArgs a;  // dx = (dz' D) A^T
  a.m = T; a.n = L.N; a.k = L.rd;
  a.A = dzp; a.sam = L.rd; a.sak = 1;
  a.kscale = Dm; a.klen = L.rd;
  a.B = A; a.sbk = 1; a.sbn = L.rd;
  a.C = dx; a.scm = L.N; a.scn = 1; a.tc = tdx;
  TT_CUDA(gemm_simt(a, st));
  GemmArgs bb;  // dA = x^T (dz' D)
  bb.m = L.N; bb.n = L.rd; bb.k = T;
  bb.A = x; bb.sam = 1; bb.sak = L.N; bb.ta = tx;
  bb.B = dzp; bb.sbk = L.rd; bb.sbn = 1;
  bb.cscale = Dm; bb.clen = L.rd;
  const int sum_mode = (L.flags & TT_DETERMINISTIC) ? kStore : kAtomic;  // kStore: whole K a thread
  bb.C = dA; bb.scm = L.rd; bb.scn = 1; bb.mode = sum_mode;
  TT_CUDA(gemm_simt(bb, st));
  GemmArgs c;  // dB = diag(D) z^T dy
  c.m = L.rd; c.n = L.M; c.k = T;
  c.A = z; c.sam = 1; c.sak = L.rd;
  c.rscale = Dm;
  c.B = dy; c.sbk = L.M; c.sbn = 1; c.tb = tdy;
  c.C = dB; c.scm = L.M; c.scn = 1; c.mode = sum_mode;
  TT_CUDA(gemm_simt(c, st));
  return TT_OK;
}

tt_status layer_backward(const LayerPlan& L, int64_t T, const void* x, int tx, const void* dy,
                         int tdy, const float* params, void* dx, int tdx, float* dparams,
                         bool acc, void* ws, const WsLayout& w, cudaStream_t st,
                         const RankStep* rank = nullptr, float* params_mut = nullptr) {
  const float* P[kMaxK];
  if (tdy == TT_DT_F32 && use_small(L, T, tx, tdx)) {
    prof_begin(kPhBwd, st);
    tt_status s = small_f32_backward(L, T, x, dy, params, dx, dparams, acc, st);
    prof_end(kPhBwd, st);
    if (s == TT_OK && rank)  // one CTA did the rest; the step is one more launch
      TT_CUDA(rank_update_launch(L, params_mut, dparams, *rank, st));
    return s;
  }
  const bool tc = use_tc(L, tx, tdx) && tdy == tx;
  if (!tc && (tx == TT_DT_E4M3 || tdy == TT_DT_E4M3)) return TT_ERR_UNSUPPORTED;
  // a forward of no tokens is a no-op that leaves nothing to reuse
  const bool reuse = (L.flags & TT_REUSE_MERGE) != 0 && T > 0;
  tt_status s = TT_OK;
  if (reuse) {
    chain_ptrs(L, params, ws, w, P);
  } else {
    prof_begin(kPhMerge, st);
    s = run_merge_forward(L, params, ws, w, P, tc, true, st);
    prof_end(kPhMerge, st);
    if (s != TT_OK) return s;
  }
  prof_begin(kPhBwd, st);
  ZeroList zl;
  if (!bwd_zero_add(&zl, L, ws, w, dparams, acc)) return TT_ERR_UNSUPPORTED;
  if (tc) {
    const void* zs = (L.flags & TT_REUSE_Z) && reuse ? static_cast<char*>(ws) + w.zs : nullptr;
    const DetSlots det = det_slots(L, ws, w);
    s = tc_backward(L, T, x, dy, dx, ws, w.tc, zl, tx == TT_DT_E4M3, zs,
                    w.det_slots ? &det : nullptr, st);
  } else {
    TT_CUDA(zero_list_memset(zl, st));
    s = simt_backward_tokens(L, T, x, tx, dy, tdy, params, P, dx, tdx, dparams, acc, ws, w, st);
  }
  prof_end(kPhBwd, st);
  if (s != TT_OK) return s;
  prof_begin(kPhMergeBwd, st);
  s = run_merge_backward(L, params, P, fptr(ws, w.dA), fptr(ws, w.dB), dparams, acc, tc,
                         tc && reuse, ws, w, st, rank, params_mut);
  prof_end(kPhMergeBwd, st);
  return s;
}

// ---- several layers on one input ---------------------------------------------
struct MultiLayout {
  WsLayout w[3];
  size_t dxp[2] = {};  // layer-by-layer backward: dx of layers 1, 2 before the sum
  size_t end = 0;
};

// The layers run on the multi-layer kernels when all of them fit the bf16
// tensor-core path (under TT_DETERMINISTIC too: per-CTA token-sum slots).
bool multi_fused(const tt_plan_s* p) {
  return p->L[0].act == TT_DT_BF16 && multi_tc_supported(p->L, p->G);
}

// One region a layer (its merges, packed operands and, fused, its z'),
// then (layer by layer) the partial dx buffers.
size_t multi_layout(const tt_plan_s* p, int64_t T, MultiLayout* m) {
  const bool fused = multi_fused(p);
  size_t off = 256;
  for (int g = 0; g < p->G; ++g)
    off = align_up(layer_layout(p->L[g], T, off, &m->w[g], false, fused), 256);
  if (!fused) {
    const size_t esz = out_dtype(p->L[0].act) == TT_DT_F32 ? 4 : 2;
    for (int g = 1; g < p->G; ++g) {
      m->dxp[g - 1] = off;
      off = align_up(off + (size_t)T * p->L[0].N * esz, 256);
    }
  }
  m->end = off;
  return off;
}

tt_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws || !aligned(ws, 256)) return TT_ERR_WORKSPACE;
  if (ws_bytes < need) return TT_ERR_WORKSPACE;
  return TT_OK;
}

bool act_aligned(const void* p) { return p && aligned(p, 16); }

}  // namespace
}  // namespace ttc

using namespace ttc;

extern "C" {

tt_status tt_default_ranks(int d, const int* in_modes, const int* out_modes, int R, int* ranks) {
  if (d < 1 || d > TT_MAX_D || !in_modes || !out_modes || !ranks || R < 1)
    return TT_ERR_INVALID_ARG;
  int s[kMaxK];
  for (int k = 0; k < d; ++k) {
    if (in_modes[k] < 1 || out_modes[k] < 1) return TT_ERR_INVALID_ARG;
    s[k] = in_modes[k];
    s[d + k] = out_modes[k];
  }
  const int K = 2 * d;
  ranks[0] = 1;
  ranks[K] = 1;
  for (int k = 1; k < K; ++k) {
    int64_t left = 1, right = 1;
    for (int i = 0; i < k; ++i) left = left * s[i] > R ? (int64_t)R + 1 : left * s[i];
    for (int i = k; i < K; ++i) right = right * s[i] > R ? (int64_t)R + 1 : right * s[i];
    int64_t v = R;
    if (left < v) v = left;
    if (right < v) v = right;
    ranks[k] = (int)v;
  }
  return TT_OK;
}

tt_status tt_plan(const tt_desc* desc, tt_plan_t** out) {
  if (!out) return TT_ERR_INVALID_ARG;
  *out = nullptr;
  LayerPlan L;
  tt_status s = build_layer(desc, &L);
  if (s != TT_OK) return s;
  if (L.act == TT_DT_E4M3 && !tc_f8_supported(L)) return TT_ERR_UNSUPPORTED;
  tt_plan_s* p = new (std::nothrow) tt_plan_s();
  if (!p) return TT_ERR_INVALID_ARG;
  p->kind = 0;
  p->L[0] = L;
  *out = p;
  return TT_OK;
}

tt_status tt_ffn_plan(const tt_desc* up, const tt_desc* down, tt_plan_t** out) {
  if (!out) return TT_ERR_INVALID_ARG;
  *out = nullptr;
  LayerPlan a, b;
  tt_status s = build_layer(up, &a);
  if (s != TT_OK) return s;
  s = build_layer(down, &b);
  if (s != TT_OK) return s;
  if (a.M != b.N || a.act != b.act || a.flags != b.flags) return TT_ERR_INVALID_ARG;
  if (a.act == TT_DT_E4M3) return TT_ERR_UNSUPPORTED;  // the FFN pair runs in bf16 or f32
  tt_plan_s* p = new (std::nothrow) tt_plan_s();
  if (!p) return TT_ERR_INVALID_ARG;
  p->kind = 1;
  p->L[0] = a;
  p->L[1] = b;
  *out = p;
  return TT_OK;
}

void tt_destroy(tt_plan_t* plan) { delete plan; }

static tt_status layout_out(const LayerPlan& L, size_t* core_off, size_t* diag_off,
                            size_t* n_floats) {
  if (!core_off || !diag_off || !n_floats) return TT_ERR_INVALID_ARG;
  for (int k = 0; k < L.K; ++k) core_off[k] = L.core_off[k];
  for (int e = 0; e < L.K - 1; ++e) diag_off[e] = L.diag_off[e];
  *n_floats = L.n_floats;
  return TT_OK;
}

tt_status tt_param_layout(const tt_plan_t* plan, size_t* core_off, size_t* diag_off,
                          size_t* n_floats) {
  if (!plan) return TT_ERR_INVALID_ARG;
  if (plan->kind == 2) {  // TT-matrix table: d cores, d-1 diagonals
    if (!core_off || !diag_off || !n_floats) return TT_ERR_INVALID_ARG;
    const TtmPlan& P = plan->ttm;
    for (int k = 0; k < P.d; ++k) core_off[k] = P.core_off[k];
    for (int k = 0; k < P.d - 1; ++k) diag_off[k] = P.diag_off[k];
    *n_floats = P.n_floats;
    return TT_OK;
  }
  return layout_out(plan->L[0], core_off, diag_off, n_floats);
}

tt_status tt_ffn_param_layout(const tt_plan_t* plan, int layer, size_t* core_off,
                              size_t* diag_off, size_t* n_floats) {
  if (!plan || plan->kind != 1 || layer < 0 || layer > 1) return TT_ERR_INVALID_ARG;
  return layout_out(plan->L[layer], core_off, diag_off, n_floats);
}

tt_status tt_workspace_size(const tt_plan_t* plan, int64_t T, size_t* bytes) {
  if (!plan || !bytes || T < 0) return TT_ERR_INVALID_ARG;
  if (plan->kind == 3) {
    MultiLayout m;
    *bytes = multi_layout(plan, T, &m);
  } else if (plan->kind == 0) {
    WsLayout w;
    *bytes = layer_layout(plan->L[0], T, 256, &w);
  } else if (plan->kind == 2) {
    if (T > 0x7FFFFFFF) return TT_ERR_INVALID_ARG;
    *bytes = ttm_workspace_bytes(plan->ttm, T);
  } else {
    FfnLayout f;
    *bytes = ffn_layout(plan, T, &f);
  }
  return TT_OK;
}

tt_status tt_forward(const tt_plan_t* plan, int64_t T, const void* x, const float* params,
                     void* y, void* ws, size_t ws_bytes, void* stream) {
  if (!plan || plan->kind != 0 || T < 0) return TT_ERR_INVALID_ARG;
  const LayerPlan& L = plan->L[0];
  if (T == 0) return TT_OK;
  if (!act_aligned(x) || !act_aligned(y) || !params || !aligned(params, 4))
    return TT_ERR_INVALID_ARG;
  WsLayout w;
  size_t need = layer_layout(L, T, 256, &w);
  tt_status s = check_ws(ws, ws_bytes, need);
  if (s != TT_OK) return s;
  return layer_forward(L, T, x, L.act, params, y, out_dtype(L.act), ws, w,
                       static_cast<cudaStream_t>(stream));
}

tt_status tt_backward(const tt_plan_t* plan, int64_t T, const void* x, const void* dy,
                      const float* params, void* dx, float* dparams, void* ws, size_t ws_bytes,
                      void* stream) {
  if (!plan || plan->kind != 0 || T < 0) return TT_ERR_INVALID_ARG;
  const LayerPlan& L = plan->L[0];
  if (!params || !dparams || !aligned(params, 4) || !aligned(dparams, 4))
    return TT_ERR_INVALID_ARG;
  if (T > 0 && (!act_aligned(x) || !act_aligned(dy) || !act_aligned(dx)))
    return TT_ERR_INVALID_ARG;
  WsLayout w;
  size_t need = layer_layout(L, T, 256, &w);
  tt_status s = check_ws(ws, ws_bytes, need);
  if (s != TT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool acc = (L.flags & TT_ACCUMULATE) != 0;
  return layer_backward(L, T, x, L.act, dy, L.act, params, dx, out_dtype(L.act), dparams, acc, ws,
                        w, st);
}

tt_status tt_backward_rank_update(const tt_plan_t* plan, int64_t T, const void* x,
                                  const void* dy, float* params, void* dx, float* dparams,
                                  const tt_rank_opts* opts, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (!plan || plan->kind != 0 || T < 0) return TT_ERR_INVALID_ARG;
  const LayerPlan& L = plan->L[0];
  RankStep r;
  if (!rank_step_from(opts, &r)) return TT_ERR_INVALID_ARG;
  if (!params || !dparams || !aligned(params, 4) || !aligned(dparams, 4))
    return TT_ERR_INVALID_ARG;
  if (T > 0 && (!act_aligned(x) || !act_aligned(dy) || !act_aligned(dx)))
    return TT_ERR_INVALID_ARG;
  WsLayout w;
  size_t need = layer_layout(L, T, 256, &w);
  tt_status s = check_ws(ws, ws_bytes, need);
  if (s != TT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool acc = (L.flags & TT_ACCUMULATE) != 0;
  return layer_backward(L, T, x, L.act, dy, L.act, params, dx, out_dtype(L.act), dparams, acc, ws,
                        w, st, &r, params);
}

tt_status tt_ffn_forward(const tt_plan_t* plan, int64_t T, const void* x,
                         const float* params_up, const float* params_down, void* y, void* ws,
                         size_t ws_bytes, void* stream) {
  if (!plan || plan->kind != 1 || T < 0) return TT_ERR_INVALID_ARG;
  if (T == 0) return TT_OK;
  if (!act_aligned(x) || !act_aligned(y) || !params_up || !params_down ||
      !aligned(params_up, 4) || !aligned(params_down, 4))
    return TT_ERR_INVALID_ARG;
  FfnLayout f;
  size_t need = ffn_layout(plan, T, &f);
  tt_status s = check_ws(ws, ws_bytes, need);
  if (s != TT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const LayerPlan& U = plan->L[0];
  const LayerPlan& D = plan->L[1];
  float* h = fptr(ws, f.h);
  float* a = fptr(ws, f.a);
  if (ffn_fused(plan)) {
    const bool reuse = (U.flags & TT_REUSE_MERGE) != 0;
    const float* P[kMaxK];
    const float* P2[kMaxK];
    prof_begin(kPhMerge, st);
    s = run_merge_forward2(U, params_up, f.up, P, D, params_down, f.down, P2, ws, reuse, st);
    prof_end(kPhMerge, st);
    if (s != TT_OK) return s;
    const bool keep = (U.flags & TT_REUSE_Z) != 0;
    prof_begin(kPhFwd, st);
    s = ffn_tc_forward(U, D, T, x, y, ws, f.up.tc, f.down.tc,
                       keep ? static_cast<char*>(ws) + f.up.zs : nullptr,
                       keep ? static_cast<char*>(ws) + f.down.zs : nullptr, true, st);
    prof_end(kPhFwd, st);
    return s;
  }
  if (ffn_tc(plan)) {
    s = layer_forward(U, T, x, TT_DT_BF16, params_up, h, TT_DT_BF16, ws, f.up, st);
    if (s != TT_OK) return s;
    prof_begin(kPhElem, st);
    TT_CUDA(gelu_fwd_bf16(T * U.M, h, a, st));
    prof_end(kPhElem, st);
    return layer_forward(D, T, a, TT_DT_BF16, params_down, y, TT_DT_BF16, ws, f.down, st);
  }
  s = layer_forward(U, T, x, U.act, params_up, h, TT_DT_F32, ws, f.up, st);
  if (s != TT_OK) return s;
  prof_begin(kPhElem, st);
  TT_CUDA(gelu_fwd(T * U.M, h, a, TT_DT_F32, st));
  prof_end(kPhElem, st);
  return layer_forward(D, T, a, TT_DT_F32, params_down, y, D.act, ws, f.down, st);
}

tt_status tt_ffn_backward(const tt_plan_t* plan, int64_t T, const void* x, const void* dy,
                          const float* params_up, const float* params_down, void* dx,
                          float* dparams_up, float* dparams_down, void* ws, size_t ws_bytes,
                          void* stream) {
  if (!plan || plan->kind != 1 || T < 0) return TT_ERR_INVALID_ARG;
  if (!params_up || !params_down || !dparams_up || !dparams_down || !aligned(params_up, 4) ||
      !aligned(params_down, 4) || !aligned(dparams_up, 4) || !aligned(dparams_down, 4))
    return TT_ERR_INVALID_ARG;
  if (T > 0 && (!act_aligned(x) || !act_aligned(dy) || !act_aligned(dx)))
    return TT_ERR_INVALID_ARG;
  FfnLayout f;
  size_t need = ffn_layout(plan, T, &f);
  tt_status s = check_ws(ws, ws_bytes, need);
  if (s != TT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const LayerPlan& U = plan->L[0];
  const LayerPlan& D = plan->L[1];
  const bool acc = (U.flags & TT_ACCUMULATE) != 0;
  float* h = fptr(ws, f.h);
  float* a = fptr(ws, f.a);
  float* da = fptr(ws, f.da);
  if (ffn_fused(plan)) {
    // the merges: the forward's (TT_REUSE_MERGE, tokens to reuse), else now
    const bool reuse = (U.flags & TT_REUSE_MERGE) != 0 && T > 0;
    const float* PU[kMaxK];
    const float* PD[kMaxK];
    if (reuse) {
      chain_ptrs(U, params_up, ws, f.up, PU);
      chain_ptrs(D, params_down, ws, f.down, PD);
    } else {
      prof_begin(kPhMerge, st);
      s = run_merge_forward2(U, params_up, f.up, PU, D, params_down, f.down, PD, ws, true, st);
      prof_end(kPhMerge, st);
      if (s != TT_OK) return s;
    }
    // z1' and z2': the forward's under TT_REUSE_Z, else computed here
    void* zs1 = static_cast<char*>(ws) + f.up.zs;
    void* zs2 = static_cast<char*>(ws) + f.down.zs;
    if (T > 0 && !((U.flags & TT_REUSE_Z) && reuse)) {
      prof_begin(kPhFwd, st);
      s = ffn_tc_forward(U, D, T, x, nullptr, ws, f.up.tc, f.down.tc, zs1, zs2, !reuse, st);
      prof_end(kPhFwd, st);
      if (s != TT_OK) return s;
    }
    prof_begin(kPhBwd, st);
    ZeroList zl;
    if (!bwd_zero_add(&zl, U, ws, f.up, dparams_up, acc) ||
        !bwd_zero_add(&zl, D, ws, f.down, dparams_down, acc))
      return TT_ERR_UNSUPPORTED;
    const DetSlots det1 = det_slots(U, ws, f.up), det2 = det_slots(D, ws, f.down);
    const bool det = f.up.det_slots && f.down.det_slots;
    s = ffn_tc_backward(U, D, T, x, dy, dx, ws, f.up.tc, f.down.tc, zs1, zs2, zl,
                        det ? &det1 : nullptr, det ? &det2 : nullptr, st);
    prof_end(kPhBwd, st);
    if (s != TT_OK) return s;
    prof_begin(kPhMergeBwd, st);
    // one launch per layer: each layer's reverse chain alone fills a wave a
    // phase, and the second launch starts as the first's CTAs leave (one
    // program of both layers measured slower: two waves a phase)
    s = run_merge_backward(D, params_down, PD, fptr(ws, f.down.dA), fptr(ws, f.down.dB),
                           dparams_down, acc, true, reuse, ws, f.down, st);
    if (s == TT_OK)
      s = run_merge_backward(U, params_up, PU, fptr(ws, f.up.dA), fptr(ws, f.up.dB), dparams_up,
                             acc, true, reuse, ws, f.up, st);
    prof_end(kPhMergeBwd, st);
    return s;
  }
  if (ffn_tc(plan)) {
    // h = up(x) and a = GELU(h) are the forward's, still in the workspace,
    // under TT_REUSE_Z (same x); otherwise they are recomputed here
    if (T > 0 && !(U.flags & TT_REUSE_Z)) {
      s = layer_forward(U, T, x, TT_DT_BF16, params_up, h, TT_DT_BF16, ws, f.up, st);
      if (s != TT_OK) return s;
      prof_begin(kPhElem, st);
      TT_CUDA(gelu_fwd_bf16(T * U.M, h, a, st));
      prof_end(kPhElem, st);
    }
    s = layer_backward(D, T, a, TT_DT_BF16, dy, TT_DT_BF16, params_down, da, TT_DT_BF16,
                       dparams_down, acc, ws, f.down, st);
    if (s != TT_OK) return s;
    if (T > 0) {
      prof_begin(kPhElem, st);
      TT_CUDA(gelu_bwd_bf16(T * U.M, h, da, st));
      prof_end(kPhElem, st);
    }
    return layer_backward(U, T, x, TT_DT_BF16, da, TT_DT_BF16, params_up, dx, TT_DT_BF16,
                          dparams_up, acc, ws, f.up, st);
  }
  if (T > 0) {
    s = layer_forward(U, T, x, U.act, params_up, h, TT_DT_F32, ws, f.up, st);
    if (s != TT_OK) return s;
    prof_begin(kPhElem, st);
    TT_CUDA(gelu_fwd(T * U.M, h, a, TT_DT_F32, st));
    prof_end(kPhElem, st);
  }
  s = layer_backward(D, T, a, TT_DT_F32, dy, D.act, params_down, da, TT_DT_F32, dparams_down,
                     acc, ws, f.down, st);
  if (s != TT_OK) return s;
  if (T > 0) {
    prof_begin(kPhElem, st);
    TT_CUDA(gelu_bwd(T * U.M, h, da, st));
    prof_end(kPhElem, st);
  }
  return layer_backward(U, T, x, U.act, da, TT_DT_F32, params_up, dx, U.act, dparams_up, acc,
                        ws, f.up, st);
}

tt_status tt_multi_plan(const tt_desc* descs, int n, tt_plan_t** out) {
  if (!out) return TT_ERR_INVALID_ARG;
  *out = nullptr;
  if (!descs || n < 1 || n > TT_MULTI_MAX) return TT_ERR_INVALID_ARG;
  LayerPlan L[TT_MULTI_MAX];
  for (int g = 0; g < n; ++g) {
    tt_status s = build_layer(&descs[g], &L[g]);
    if (s != TT_OK) return s;
    if (L[g].act != L[0].act || L[g].flags != L[0].flags || L[g].d != L[0].d)
      return TT_ERR_INVALID_ARG;
    for (int k = 0; k < L[0].d; ++k)
      if (descs[g].in_modes[k] != descs[0].in_modes[k]) return TT_ERR_INVALID_ARG;
    if (L[g].act == TT_DT_E4M3 && !tc_f8_supported(L[g])) return TT_ERR_UNSUPPORTED;
  }
  tt_plan_s* p = new (std::nothrow) tt_plan_s();
  if (!p) return TT_ERR_INVALID_ARG;
  p->kind = 3;
  p->G = n;
  for (int g = 0; g < n; ++g) p->L[g] = L[g];
  *out = p;
  return TT_OK;
}

tt_status tt_multi_param_layout(const tt_plan_t* plan, int layer, size_t* core_off,
                                size_t* diag_off, size_t* n_floats) {
  if (!plan || plan->kind != 3 || layer < 0 || layer >= plan->G) return TT_ERR_INVALID_ARG;
  return layout_out(plan->L[layer], core_off, diag_off, n_floats);
}

tt_status tt_multi_forward(const tt_plan_t* plan, int64_t T, const void* x,
                           const float* const* params, void* const* y, void* ws,
                           size_t ws_bytes, void* stream) {
  if (!plan || plan->kind != 3 || T < 0 || !params || !y) return TT_ERR_INVALID_ARG;
  const int G = plan->G;
  for (int g = 0; g < G; ++g)
    if (!params[g] || !aligned(params[g], 4)) return TT_ERR_INVALID_ARG;
  if (T == 0) return TT_OK;
  if (!act_aligned(x)) return TT_ERR_INVALID_ARG;
  for (int g = 0; g < G; ++g)
    if (!act_aligned(y[g])) return TT_ERR_INVALID_ARG;
  MultiLayout m;
  tt_status s = check_ws(ws, ws_bytes, multi_layout(plan, T, &m));
  if (s != TT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int act = plan->L[0].act;
  if (!multi_fused(plan)) {
    for (int g = 0; g < G && s == TT_OK; ++g)
      s = layer_forward(plan->L[g], T, x, act, params[g], y[g], out_dtype(act), ws, m.w[g], st);
    return s;
  }
  const bool reuse = (plan->L[0].flags & TT_REUSE_MERGE) != 0;
  const bool keep = (plan->L[0].flags & TT_REUSE_Z) != 0;
  const LayerPlan* Ls[TT_MULTI_MAX];
  const WsLayout* wl[TT_MULTI_MAX];
  const float* P[TT_MULTI_MAX][kMaxK];
  const float** Pp[TT_MULTI_MAX];
  void* zs[TT_MULTI_MAX];
  size_t offs[TT_MULTI_MAX];
  for (int g = 0; g < G; ++g) {
    Ls[g] = &plan->L[g];
    wl[g] = &m.w[g];
    Pp[g] = P[g];
    zs[g] = static_cast<char*>(ws) + m.w[g].zs;
    offs[g] = m.w[g].tc;
  }
  prof_begin(kPhMerge, st);
  s = run_merge_forward_n(G, Ls, params, wl, Pp, ws, reuse, st);
  prof_end(kPhMerge, st);
  if (s != TT_OK) return s;
  prof_begin(kPhFwd, st);
  s = multi_tc_forward(plan->L, G, T, x, y, ws, offs, keep ? zs : nullptr, true, st);
  prof_end(kPhFwd, st);
  return s;
}

tt_status tt_multi_backward(const tt_plan_t* plan, int64_t T, const void* x,
                            const void* const* dy, const float* const* params, void* dx,
                            float* const* dparams, void* ws, size_t ws_bytes, void* stream) {
  if (!plan || plan->kind != 3 || T < 0 || !params || !dparams || !dy)
    return TT_ERR_INVALID_ARG;
  const int G = plan->G;
  for (int g = 0; g < G; ++g) {
    if (!params[g] || !dparams[g] || !aligned(params[g], 4) || !aligned(dparams[g], 4))
      return TT_ERR_INVALID_ARG;
    if (T > 0 && !act_aligned(dy[g])) return TT_ERR_INVALID_ARG;
  }
  if (T > 0 && (!act_aligned(x) || !act_aligned(dx))) return TT_ERR_INVALID_ARG;
  MultiLayout m;
  tt_status s = check_ws(ws, ws_bytes, multi_layout(plan, T, &m));
  if (s != TT_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int act = plan->L[0].act;
  const bool acc = (plan->L[0].flags & TT_ACCUMULATE) != 0;
  if (!multi_fused(plan)) {
    // layer by layer: layer 0's dx into dx, the others' beside it, then the sum
    const void* parts[TT_MULTI_MAX - 1];
    for (int g = 0; g < G && s == TT_OK; ++g) {
      void* dxg = g == 0 ? dx : static_cast<char*>(ws) + m.dxp[g - 1];
      if (g > 0) parts[g - 1] = dxg;
      s = layer_backward(plan->L[g], T, x, act, dy[g], act, params[g], dxg, out_dtype(act),
                         dparams[g], acc, ws, m.w[g], st);
    }
    if (s != TT_OK || T == 0 || G == 1) return s;
    prof_begin(kPhElem, st);
    TT_CUDA(sum_into(T * plan->L[0].N, dx, parts, G - 1, out_dtype(act), st));
    prof_end(kPhElem, st);
    return TT_OK;
  }
  // the merges: the forward's (TT_REUSE_MERGE, tokens to reuse), else now
  const bool reuse = (plan->L[0].flags & TT_REUSE_MERGE) != 0 && T > 0;
  const LayerPlan* Ls[TT_MULTI_MAX];
  const WsLayout* wl[TT_MULTI_MAX];
  const float* P[TT_MULTI_MAX][kMaxK];
  const float** Pp[TT_MULTI_MAX];
  void* zs[TT_MULTI_MAX];
  size_t offs[TT_MULTI_MAX];
  ZeroList zl;
  for (int g = 0; g < G; ++g) {
    Ls[g] = &plan->L[g];
    wl[g] = &m.w[g];
    Pp[g] = P[g];
    zs[g] = static_cast<char*>(ws) + m.w[g].zs;
    offs[g] = m.w[g].tc;
    if (!bwd_zero_add(&zl, plan->L[g], ws, m.w[g], dparams[g], acc)) return TT_ERR_UNSUPPORTED;
  }
  if (reuse) {
    for (int g = 0; g < G; ++g) chain_ptrs(plan->L[g], params[g], ws, m.w[g], P[g]);
  } else {
    prof_begin(kPhMerge, st);
    s = run_merge_forward_n(G, Ls, params, wl, Pp, ws, true, st);
    prof_end(kPhMerge, st);
    if (s != TT_OK) return s;
  }
  // every z'_g: the forward's under TT_REUSE_Z, else computed here
  if (T > 0 && !((plan->L[0].flags & TT_REUSE_Z) && reuse)) {
    prof_begin(kPhFwd, st);
    s = multi_tc_forward(plan->L, G, T, x, nullptr, ws, offs, zs, !reuse, st);
    prof_end(kPhFwd, st);
    if (s != TT_OK) return s;
  }
  prof_begin(kPhBwd, st);
  DetSlots det[TT_MULTI_MAX];
  bool use_det = true;
  for (int g = 0; g < G; ++g) {
    det[g] = det_slots(plan->L[g], ws, m.w[g]);
    use_det &= m.w[g].det_slots > 0;
  }
  s = multi_tc_backward(plan->L, G, T, x, dy, dx, ws, offs, zs, zl, use_det ? det : nullptr, st);
  prof_end(kPhBwd, st);
  if (s != TT_OK) return s;
  prof_begin(kPhMergeBwd, st);
  // the layers' programs in one launch where they fit one (a launch each
  // otherwise, or with TTC_MULTI_MERGE_SPLIT=1, a measurement aid)
  static int split = -1;
  if (split < 0) {
    const char* e = getenv("TTC_MULTI_MERGE_SPLIT");
    split = (e && e[0] && e[0] != '0') ? 1 : 0;
  }
  s = TT_ERR_UNSUPPORTED;
  if (!split && G > 1) {
    MergeBwd* mb[TT_MULTI_MAX] = {};
    alignas(MergeBwd) unsigned char store[TT_MULTI_MAX][sizeof(MergeBwd)];
    for (int g = 0; g < G; ++g)
      mb[g] = new (store[g]) MergeBwd(plan->L[g], params[g], P[g], fptr(ws, m.w[g].dA),
                                      fptr(ws, m.w[g].dB), dparams[g], acc, true, reuse, ws,
                                      m.w[g]);
    s = run_merge_backward_multi(mb, G, st);
    for (int g = 0; g < G; ++g) mb[g]->~MergeBwd();
  }
  if (s == TT_ERR_UNSUPPORTED) {  // nothing was launched
    s = TT_OK;
    for (int g = 0; g < G && s == TT_OK; ++g)
      s = run_merge_backward(plan->L[g], params[g], P[g], fptr(ws, m.w[g].dA),
                             fptr(ws, m.w[g].dB), dparams[g], acc, true, reuse, ws, m.w[g], st);
  }
  prof_end(kPhMergeBwd, st);
  return s;
}

tt_status tt_get_device_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return TT_ERR_CUDA;
  DeviceStatus h{0, 0}, e{0, 0};
  if (read_and_clear_device_status(&h) != cudaSuccess) return TT_ERR_CUDA;
  if (read_and_clear_ttm_status(&e) != cudaSuccess) return TT_ERR_CUDA;
  if (h.code == TT_ERR_TIMEOUT) return TT_ERR_TIMEOUT;
  if (h.code != 0 || e.code != 0) return TT_ERR_DEVICE;
  return TT_OK;
}

const char* tt_status_string(tt_status s) {
  switch (s) {
    case TT_OK: return "TT_OK";
    case TT_ERR_INVALID_ARG: return "TT_ERR_INVALID_ARG: invalid argument";
    case TT_ERR_UNSUPPORTED: return "TT_ERR_UNSUPPORTED: no kernel for this layer";
    case TT_ERR_WORKSPACE: return "TT_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case TT_ERR_CUDA: return "TT_ERR_CUDA: CUDA call or launch failed";
    case TT_ERR_TIMEOUT: return "TT_ERR_TIMEOUT: a bounded device wait ran out";
    case TT_ERR_DEVICE: return "TT_ERR_DEVICE: device-side check failed";
  }
  return "unknown tt_status";
}

}  // extern "C"
