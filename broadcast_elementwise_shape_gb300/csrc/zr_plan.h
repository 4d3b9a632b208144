// zr_plan.h — host planner: validation, broadcast, dimension coalescing and
// construction of the by-value kernel plans.  Pure host C++; the launches
// live in the .cu files.
#pragma once

#include <stdint.h>
#include <stddef.h>
#include <string>

#include "../../include/zr.h"
#include "zr_internal.h"

namespace zr {

// A validated tensor view with explicit strides.
struct TDesc {
  const float* ptr = nullptr;
  int nd = 0;
  int64_t size[kMaxDims] = {};
  int64_t stride[kMaxDims] = {};
  int64_t numel = 1;
  int64_t extent = 0;  // largest element offset + 1 (0 when empty)
};

int read_tensor(const zr_tensor& t, TDesc* d);
int broadcast_sizes(int nda, const int64_t* sa, int ndb, const int64_t* sb, int* nd,
                    int64_t* so);
void contiguous_strides(int nd, const int64_t* size, int64_t* stride);

// Operand slots while coalescing: G/A/B/D as in zr_internal.h plus the two
// gradient index maps (dense in a's / b's shape, 0 on broadcast dims).
constexpr int kSlotXA = 4;
constexpr int kSlotXB = 5;
constexpr int kProbSlots = 6;

// The output index space after dropping size-1 dims and merging adjacent
// dims that every active operand walks contiguously; row-major, dims[0]
// outermost.
struct Prob {
  int n = 0;
  int64_t size[kMaxDims] = {};
  int64_t st[kProbSlots][kMaxDims] = {};
  uint32_t active = 0;  // bit k: slot k takes part
  int es = 4;           // bytes per stored element: 4 (float) or 2 (bfloat16)
};

// Strides of x against an output of rank n: 0 where x is missing or 1.
void align_strides(const TDesc& x, int n, const int64_t* out_size, int64_t* st);
// Row-major strides of x's own shape against the output: 0 on broadcast dims.
void grad_index_strides(const TDesc& x, int n, const int64_t* out_size, int64_t* st);

// Drop size-1 dims, optionally sort by descending stride of `order_slot`
// (-1 = keep order), and merge.  Splits an innermost dim that is too long for
// 32-bit column indexing.  Returns ZR_OK or ZR_ERR_SIZE.
int coalesce(int n, const int64_t* size, const int64_t (*st)[kMaxDims], uint32_t active,
             int order_slot, Prob* P);

struct EwBuild {
  EwPlan plan;
  int vec;
  int es;             // bytes per stored element (Prob::es)
  bool uni1 = false;  // input slot 1 is one element (a forward's b with numel 1)
  bool gelu_tab = false;  // bfloat16 GeLU by table (k_gelu_bf16, grid in plan.n_cta)
};
// Elementwise plan over P with input slots 0..2 and output slot 3.
// occ: resident CTAs per SM of the kernel that will run the plan.
// Second-pass layout for the partial pointer now set in c: 4 outputs per
// thread with 16-byte partial loads when nout is a multiple of 4, at least
// 64 per SM (so the groups of 4 still fill the GPU), and the partials are
// 16-byte aligned.
void combine_vectorize(CombinePlan* c);
// Thread blocks of the second pass.
uint64_t combine_blocks(const CombinePlan& c);
// Dynamic shared memory of a reduction pass: its row-offset table, its tree
// and `stages` staged batches of `stage_ns` streamed inputs.
uint64_t red_smem_bytes(const RedPlan& p, int vec, uint32_t stages, uint32_t stage_ns);
int build_ew(const Prob& P, const float* const in[3], float* const out[2], uint32_t read_mask,
             uint32_t stream_mask, int occ, EwBuild* eb);

// Transposed-input forward plan; ZR_OK when the layout qualifies, 1 if not.
int build_tr(const Prob& P, const float* a, const float* b, float* out, TrPlan* tp);
std::string describe_tr(const TrPlan& tp);

struct RedBuild {
  RedPlan plan;
  CombinePlan comb;
  int vec;
  size_t ws_bytes;  // partial workspace (0 when nslots == 1); partials are binary32
  int es;           // bytes per stored element (Prob::es)
};
// Reduction plan over P for the gradient whose index map is slot `xslot`.
// `d_out` (may be null) is written densely from slot 3 offsets.
// vec_override: 0 = choose VEC from alignment; 1 or 4 = size the tiling as if
// VEC were that value (used to report a workspace size that holds whatever
// the alignment of the run-time pointers turns out to be).
// occ: resident CTAs per SM of the kernel that will run the plan;
// occ_cl_kept / occ_cl_red: the same for the cluster variant with the inner
// dim kept / reduced (0: no cluster plan).
// post: X's total is multiplied by a per-output factor (division's -1/b^2
// for grad_b); with partial slots the workspace also holds those factors,
// one per output after the slots, and the second pass applies them.
int build_red(const Prob& P, int xslot, const float* g, const float* a, const float* b,
              uint32_t read_mask, uint32_t stream_mask, float* x_out, float* d_out,
              int vec_override, int occ, int occ_cl_kept, int occ_cl_red, RedBuild* rb,
              bool post = false);

struct ChainBuild {
  ChainPlan plan;
  CombinePlan comb_b, comb_c;
  size_t ws_b_bytes, ws_c_bytes;  // grad_b / grad_c partial regions (0: none)
};
// Fused chain backward plan over P (slots G, A, B, D = grad_a, XB = grad_b's
// index map).  Returns ZR_OK when the layout qualifies (16-byte vectors, b
// reduced with its inner dim kept; c with b's dense layout, or one element),
// 1 when it does not, or an error code.  vec_override as for build_red.
// div1 / div2: op1 / op2 is a division, whose -1/b^2 (-1/c^2) factor the
// second passes apply to each total (the workspace holds the factors).
int build_chain(const Prob& P, const float* g, const float* a, const float* b, const float* c,
                bool c_scalar, float* grad_a, float* grad_b, float* grad_c, uint32_t stream_mask,
                int vec_override, ChainBuild* cb, bool div1, bool div2);
std::string describe_chain(const ChainBuild& cb);

struct SabBuild {
  SabPlan plan;
  CombinePlan comb_a, comb_b;
  int rpt;                  // rows per thread (ta * nvc / 256)
  size_t ws_a_bytes, ws_b_bytes;
};
// Fused both-reduced plan; returns ZR_OK when the shape qualifies, 1 when it
// does not (the caller then runs one reduction pass per gradient), or an
// error code.  post: grad_b's totals carry a per-output factor (division),
// stored after grad_b's slots and applied by its second pass.
int build_sab(const Prob& P, const float* g, const float* a, const float* b, float* grad_a,
              float* grad_b, uint32_t read_mask, SabBuild* sb, bool post);

// Split forward plan (SabFPlan); ZR_OK when the layout qualifies, 1 if not.
// Slots of P: 0 = a, 1 = b, 3 = out.
int build_sabf(const Prob& P, const float* a, const float* b, float* out, SabFPlan* sp, int* rpt);
std::string describe_sabf(const SabFPlan& sp, int rpt);

std::string describe_ew(const EwBuild& eb);
std::string describe_sab(const SabBuild& sb);
std::string describe_red(const RedBuild& rb);

}  // namespace zr
