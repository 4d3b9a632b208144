// zr_launch_ew.cu — instantiations and launches of the elementwise kernel.
#include "zr_launch.h"
#include "zr_kernels.cuh"

namespace zr {

namespace {

template <class F, int NOUT>
cudaError_t launch_ew_t(const EwBuild& eb, cudaStream_t s, bool dry) {
  // Refuse a launch whose kernel would dereference a missing operand.
  if (!eb.plan.in[0] || (F::kR1 && !eb.plan.in[1]) || (F::kR2 && !eb.plan.in[2]) ||
      (!eb.plan.out[0] && !eb.plan.out[1]))
    return cudaErrorInvalidValue;
  if (dry) return cudaSuccess;
  if (eb.vec == 4) return launch_ew_kernel<F, 4, NOUT>(eb.plan, s);
  return launch_ew_kernel<F, 1, NOUT>(eb.plan, s);
}

template <int OP>
cudaError_t launch_direct_op(int want, const EwBuild& eb, cudaStream_t s, bool dry) {
  switch (want) {
    case 1: return launch_ew_t<BwdDirectF<OP, 1>, 2>(eb, s, dry);
    case 2: return launch_ew_t<BwdDirectF<OP, 2>, 2>(eb, s, dry);
    default: return launch_ew_t<BwdDirectF<OP, 3>, 2>(eb, s, dry);
  }
}

}  // namespace

cudaError_t launch_fwd(int op, const EwBuild& eb, cudaStream_t s, bool dry) {
  if (eb.es == 2) return launch_fwd_bf16(op, eb, s, dry);
  switch (op) {
    case OP_ADD: return launch_ew_t<FwdF<OP_ADD>, 1>(eb, s, dry);
    case OP_SUB: return launch_ew_t<FwdF<OP_SUB>, 1>(eb, s, dry);
    case OP_MUL: return launch_ew_t<FwdF<OP_MUL>, 1>(eb, s, dry);
    default:
      return eb.uni1 ? launch_ew_t<FwdF<OP_DIV, false, true>, 1>(eb, s, dry)
                     : launch_ew_t<FwdF<OP_DIV>, 1>(eb, s, dry);
  }
}

namespace {
template <int OP>
cudaError_t launch_sabf_op(int rpt, const SabFPlan& sp, cudaStream_t s) {
  switch (rpt) {
    case 1: return launch_k(k_sabf<OP, 1>, sp.n_cta, kThreads, 0, s, sp);
    case 2: return launch_k(k_sabf<OP, 2>, sp.n_cta, kThreads, 0, s, sp);
    case 4: return launch_k(k_sabf<OP, 4>, sp.n_cta, kThreads, 0, s, sp);
    case 8: return launch_k(k_sabf<OP, 8>, sp.n_cta, kThreads, 0, s, sp);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

cudaError_t launch_fwd_sabf(int op, int rpt, const SabFPlan& sp, cudaStream_t s, bool dry) {
  if (!sp.a || !sp.b || !sp.out || (rpt != 1 && rpt != 2 && rpt != 4 && rpt != 8))
    return cudaErrorInvalidValue;
  if (dry) return cudaSuccess;
  switch (op) {
    case OP_ADD: return launch_sabf_op<OP_ADD>(rpt, sp, s);
    case OP_SUB: return launch_sabf_op<OP_SUB>(rpt, sp, s);
    case OP_MUL: return launch_sabf_op<OP_MUL>(rpt, sp, s);
    default: return launch_sabf_op<OP_DIV>(rpt, sp, s);
  }
}

cudaError_t launch_fwd_tr(int op, const TrPlan& tp, cudaStream_t s, bool dry) {
  if (!tp.x || !tp.y || !tp.out) return cudaErrorInvalidValue;
  if (dry) return cudaSuccess;
  switch (op) {
    case OP_ADD: return launch_k(k_transpose<OP_ADD>, tp.n_cta, kThreads, 0, s, tp);
    case OP_SUB: return launch_k(k_transpose<OP_SUB>, tp.n_cta, kThreads, 0, s, tp);
    case OP_MUL: return launch_k(k_transpose<OP_MUL>, tp.n_cta, kThreads, 0, s, tp);
    default: return launch_k(k_transpose<OP_DIV>, tp.n_cta, kThreads, 0, s, tp);
  }
}

cudaError_t launch_bwd_direct(int op, int want, const EwBuild& eb, cudaStream_t s, bool dry) {
  if (eb.es == 2) return launch_bwd_direct_bf16(op, want, eb, s, dry);
  switch (op) {
    case OP_ADD: return launch_direct_op<OP_ADD>(want, eb, s, dry);
    case OP_SUB: return launch_direct_op<OP_SUB>(want, eb, s, dry);
    case OP_MUL: return launch_direct_op<OP_MUL>(want, eb, s, dry);
    default: return launch_direct_op<OP_DIV>(want, eb, s, dry);
  }
}

cudaError_t launch_copy(const EwBuild& eb, cudaStream_t s, bool dry) {
  if (eb.es == 2) return launch_copy_bf16(eb, s, dry);
  return launch_ew_t<CopyF, 1>(eb, s, dry);
}

cudaError_t launch_unary_fwd(int uop, const EwBuild& eb, cudaStream_t s, bool dry) {
  if (eb.es == 2) return launch_unary_fwd_bf16(uop, eb, s, dry);
  return uop == UN_SCALE ? launch_ew_t<UnaryF<UN_SCALE>, 1>(eb, s, dry)
                         : launch_ew_t<UnaryF<UN_GELU>, 1>(eb, s, dry);
}

cudaError_t launch_unary_bwd(int uop, const EwBuild& eb, cudaStream_t s, bool dry) {
  if (eb.es == 2) return launch_unary_bwd_bf16(uop, eb, s, dry);
  return uop == UN_SCALE ? launch_ew_t<UnaryBwdF<UN_SCALE>, 1>(eb, s, dry)
                         : launch_ew_t<UnaryBwdF<UN_GELU>, 1>(eb, s, dry);
}

cudaError_t occupancy_ew(int which, int* planned, int* actual) {
  const size_t smem = size_t(kMaxTileRows) * kMaxOperands * sizeof(int64_t);
  switch (which) {
    case 0:
      *planned = kOccEwFwd;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_elementwise<FwdF<OP_ADD>, 4, 1>,
                                                           kThreads, smem);
    case 1:
      *planned = kOccEwFwd;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_elementwise<FwdF<OP_DIV>, 4, 1>,
                                                           kThreads, smem);
    case 2:
      *planned = kOccEwBwd;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_elementwise<BwdDirectF<OP_DIV, 3>, 4, 2>, kThreads, smem);
    case 3:
      *planned = kOccEwCopy;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_elementwise<CopyF, 4, 1>,
                                                           kThreads, smem);
    case 4:
      *planned = kOccGeluFwd;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_elementwise<UnaryF<UN_GELU>, 4, 1>,
                                                           kThreads, smem);
    case 5:
      *planned = kOccEwFwd;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_elementwise<UnaryBwdF<UN_GELU>, 4, 1>, kThreads, smem);
    // The flat kernel (no shared memory): forward add, float GeLU forward.
    case 6:
      *planned = kOccEwFwd;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_flat<FwdF<OP_ADD>, 4, 1>,
                                                           kThreads, 0);
    case 7:
      *planned = kOccGeluFwd;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_flat<UnaryF<UN_GELU>, 4, 1>,
                                                           kThreads, 0);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t occupancy_other(int which, int* planned, int* actual) {
  switch (which) {
    case 0:
      *planned = kOccSabf;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_sabf<OP_DIV, 8>, kThreads, 0);
    case 1:
      *planned = kOccTr;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_transpose<OP_SUB>, kThreads, 0);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace zr
