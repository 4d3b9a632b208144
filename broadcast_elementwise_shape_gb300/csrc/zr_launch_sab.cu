// zr_launch_sab.cu — instantiations and launches of the fused both-reduced
// backward (k_sab) and its two combine passes.
#include "zr_launch.h"
#include "zr_sab.cuh"

namespace zr {

namespace {

template <int OP, int RPT>
cudaError_t launch_sab_t(const SabBuild& sb, cudaStream_t s, bool dry) {
  const SabPlan& p = sb.plan;
  constexpr bool kUses = OP == OP_MUL || OP == OP_DIV;
  if (!p.g || (kUses && (!p.a || !p.b)) || !p.ws_a || !p.ws_b || !sb.comb_a.out ||
      !sb.comb_b.out)
    return cudaErrorInvalidValue;
  // Division stores grad_b's factors after its slots: only a plan sized for
  // them may run.
  if (OP == OP_DIV && !sb.comb_b.post) return cudaErrorInvalidValue;
  if (dry) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k_sab<OP, RPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(p.smem_bytes));
  if (e != cudaSuccess) return e;
  e = launch_k(k_sab<OP, RPT>, p.grid, kSabThreads, p.smem_bytes, s, p);
  if (e != cudaSuccess) return e;
  CombinePlan ca = sb.comb_a, cb = sb.comb_b;
  ca.partial = p.ws_a;
  cb.partial = p.ws_b;
  e = launch_combine_f32(ca, s);
  if (e != cudaSuccess) return e;
  return launch_combine_f32(cb, s);
}

template <int OP>
cudaError_t launch_sab_op(const SabBuild& sb, cudaStream_t s, bool dry) {
  switch (sb.rpt) {
    case 1: return launch_sab_t<OP, 1>(sb, s, dry);
    case 2: return launch_sab_t<OP, 2>(sb, s, dry);
    case 4: return launch_sab_t<OP, 4>(sb, s, dry);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_sab(int op, const SabBuild& sb, cudaStream_t s, bool dry) {
  switch (op) {
    case OP_ADD: return launch_sab_op<OP_ADD>(sb, s, dry);
    case OP_SUB: return launch_sab_op<OP_SUB>(sb, s, dry);
    case OP_MUL: return launch_sab_op<OP_MUL>(sb, s, dry);
    default: return launch_sab_op<OP_DIV>(sb, s, dry);
  }
}

}  // namespace zr
