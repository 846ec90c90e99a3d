// One-launch execution of the T-independent merge work (chain merges, their
// reverse, operand packing, gradient unpacking): a persistent cooperative
// kernel walks a short list of phases; the tasks of one phase are spread
// over all CTAs and a bounded grid barrier separates phases.
#pragma once

#include "rank_step.cuh"
#include "tc_fused.h"
#include "ttc_internal.h"

namespace ttc {

enum EngKind {
  kEGemm = 0,      // C (op)= ... (GemmArgs); split-K partials when splits > 1
  kEGemmFinal = 1, // sum split-K partials, apply scales, store/accumulate into C
  kEColdot = 2,    // out[c] (=|+=) sum_u X[u,c] Y[u,c] (masked by D == 0)
  kEScale = 3,     // out[i] (=|+=) in[i] * scale[i % len]
  kEPack = 4,      // tensor-core operands from A, B, D_d (+ zero gradient sums)
  kEUnpack = 5,    // compacted gradient sums -> dA, dB, dD_d
  kEDd = 6,        // compacted dD_d sum -> dD_d only
  kEChain = 7,     // rows of one side's merged chain, recomputed per prefix
  kERank = 8       // the rank-adaptive step over one layer's packed parameters
};

// One side of the chain for kEChain: cores C_0..C_{L-1} (C_k of shape
// (r[k], s[k], r[k+1]), r[0] the left boundary), diagonals E_k between C_k
// and C_{k+1}.  A prefix is (alpha, s_0..s_{L-2}); its P_k rows and the
// s_{L-1} final rows of P_{L-1} (= A or B) are written.
struct ChainDesc {
  const float* core[TT_MAX_D] = {};
  const float* diag[TT_MAX_D] = {};
  float* prow[TT_MAX_D] = {};   // P_k buffers for 1 <= k <= L-2
  float* out = nullptr;         // P_{L-1} (null: packed operands only)
  int r[TT_MAX_D + 1] = {};
  int s[TT_MAX_D] = {};
  int L = 0;
  int pb = 1;                   // prefixes per unit
  int sb = 1;                   // last-mode indices per unit
  int nsb = 1;                  // number of last-mode blocks
  int64_t nprefix = 0;
};

struct alignas(16) EngTask {
  int kind = 0;
  int units = 0;
  int splits = 1;       // kEGemm / kEGemmFinal
  int tm = 32, tn = 32; // kEGemm output tile (16 or 32 each)
  int tiles_n = 1;      // kEGemm: tiles along n
  int kchunk = 0;       // kEGemm: K extent of one split
  int atomic_splits = 0;  // kEGemm: K splits may add into C (mode kAtomic)
  int64_t pcap = 0;     // kEGemm: floats of the split-K partial buffer `partial`
  // kEGemm: division by splits and by tiles_n as a multiply and a shift
  // (x / d == (x * mul) >> sh for 0 <= x < 2^31)
  unsigned long long div_s_mul = 0, div_n_mul = 0;
  int div_s_sh = 0, div_n_sh = 0;
  GemmArgs g;           // kEGemm / kEGemmFinal
  float* partial = nullptr;  // split-K partials [splits][m][n]
  // kEColdot / kEScale / pack / unpack operands
  const float* x = nullptr;
  const float* y = nullptr;
  const float* s = nullptr;
  float* out = nullptr;
  int64_t n = 0, sx = 0, sy = 0;
  int len = 1, acc = 0;
  int chunk = 1024;     // kEScale, kERank, kEPack, kEUnpack: elements per unit
  // pack / unpack (s = middle diagonal D_d, out = dD_d for unpack)
  const float* A = nullptr;
  const float* B = nullptr;
  TcPtrs tc;
  float* dA = nullptr;
  float* dB = nullptr;
  int rd = 0, N = 0, M = 0, zero = 0;
  // kEGemm extras for the tensor-core path:
  //  pack_side 1/2: the GEMM computes A (N x rd) / B (rd x M); its epilogue
  //    also writes the compacted bf16 operands (tc, compaction from s = D_d).
  //  gather 1/2: the operand that reads dA / dB (gather_op 0 = A, 1 = B)
  //    reads the compacted token sums tc.dAc / tc.dBc instead.
  int pack_side = 0, gather = 0, gather_op = 0, pad_only = 0;
  //  fold_g: the GEMM is the last reverse step of a side, C = dQ is not
  //    stored; each output v (row, c) adds v * cscale[c] to fold_g (the
  //    first core's gradient, laid out like C) and fold_p[row, c] * v to
  //    fold_dd[c] (dD of the first link, skipped where cscale[c] == 0).
  float* fold_g = nullptr;
  const float* fold_p = nullptr;
  float* fold_dd = nullptr;
  ChainDesc ch;  // kEChain (pack_side selects the packing, s = D_d)
  RankStep rk;   // kERank: out = params, dA = dparams, n = floats, len = core floats
};

constexpr int kEngMaxTasks = 46;  // two order-6 layers (an FFN pair) in one program
constexpr int kEngMaxPhases = 8;

struct alignas(16) EngProgram {
  int ntasks = 0, nphases = 0;
  // Grid-barrier arrival counter of this call (a 64-bit word on its own
  // 256-byte line of the caller's workspace).  A program of more than one
  // phase needs it, zeroed in stream order before the launch; every call
  // has its own, so calls on different streams with different workspaces
  // never share one.
  unsigned long long* bar = nullptr;
  int phase_begin[kEngMaxPhases + 1] = {};
  // units of a phase are dealt in this task order (set by eng_launch: the
  // tasks with the costliest units first)
  unsigned char order[kEngMaxTasks] = {};
  // set by eng_launch: the units of a phase dealt before order position i
  // (ustart), and every phase's units (ptotal), so that a CTA finds its
  // unit's task in a few reads of adjacent words instead of a walk through
  // the task records
  int ustart[kEngMaxTasks] = {};
  int ptotal[kEngMaxPhases] = {};
  EngTask t[kEngMaxTasks];
};

// Builders used by the host code (ttc_api.cu).
struct EngBuilder {
  EngProgram p;
  bool overflow = false;
  void begin_phase();  // also balances the phase before it
  EngTask* add();
  void end();  // closes (and balances) the last phase
  // Narrows the GEMM tasks of the last phase (larger tiles, fewer K splits)
  // until its units fit the fewest waves of `budget` CTAs that its
  // narrowest configuration allows (one wave where possible).
  void balance(int budget);
  // After balance, for a phase of one wave: lowers its costliest unit.
  void refine(int budget);
  // After balance, for a phase of several waves: shortens it as dealt.
  void refine_waves();
};

// Units for a GEMM task of the engine's tile size and a split-K count.
// atomic_splits: a kAtomic GEMM may be split along K, every split adding
// into C (which must be zero before the phase).  The tile and split choice
// takes the most units up to max_units (EngBuilder::balance narrows it).
void eng_gemm_task(EngTask* t, const GemmArgs& g, float* partial_ws, size_t partial_cap,
                   bool atomic_splits = false, int max_units = 128);
// SMs of the current device (the engine's grid), cached after the first call.
int eng_sm_count();
void eng_gemm_final_task(EngTask* t, const EngTask& gemm);
// false when the chain does not fit the unit's shared-memory staging
bool eng_chain_task(EngTask* t, const ChainDesc& c);
void eng_pack_task(EngTask* t, const LayerPlan& L, const float* A, const float* B,
                   const float* Dmid, const TcPtrs& tc, bool zero_grads, bool pad_only = false);
void eng_dd_task(EngTask* t, const LayerPlan& L, const TcPtrs& tc, const float* Dmid,
                 float* dDout, bool acc);
void eng_unpack_task(EngTask* t, const LayerPlan& L, const TcPtrs& tc, const float* Dmid,
                     float* dA, float* dB, float* dDout, bool acc);
// The rank-adaptive step (rank_step_elem) over the packed params / dparams.
void eng_rank_task(EngTask* t, const LayerPlan& L, float* params, float* dparams,
                   const RankStep& r);

// Launch (cooperative when it has more than one phase: one CTA per SM).
// Returns cudaSuccess or the error; cudaErrorInvalidValue for a program of
// several phases without a barrier counter.
cudaError_t eng_launch(const EngProgram& p, cudaStream_t st);

// Bytes of split-K partial scratch a GEMM of this shape may use.
size_t eng_partial_floats(int64_t m, int64_t n, int64_t k);

}  // namespace ttc
