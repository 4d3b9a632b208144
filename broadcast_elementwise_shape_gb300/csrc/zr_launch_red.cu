// zr_launch_red.cu — instantiations and launches of the reduction and
// combine kernels.
#include "zr_launch.h"
#include "zr_kernels.cuh"

namespace zr {

namespace {

template <int OP, int WHICH>
cudaError_t launch_red_t(const RedBuild& rb, cudaStream_t s, bool dry) {
  const RedPlan& p = rb.plan;
  // Refuse a launch whose kernel would dereference an operand the plan did
  // not provide.
  const bool has_d = p.d_out != nullptr;
  if (!p.g || (RedTerms<OP, WHICH>::reads_a(has_d) && !p.a) ||
      (RedTerms<OP, WHICH>::reads_b(has_d) && !p.b) || !p.x_final ||
      (p.nslots > 1 && !p.partial))
    return cudaErrorInvalidValue;
  if (p.cluster > 1 && (rb.vec != 4 || p.nslots != 1 || p.n_cta % p.cluster != 0 ||
                        p.cluster > kMaxCluster))
    return cudaErrorInvalidValue;
  // With partial slots, division's grad_b stores its factors after the slots:
  // only a plan whose workspace was sized for them may run.
  if (RedTerms<OP, WHICH>::kPost && p.nslots > 1 && !rb.comb.post) return cudaErrorInvalidValue;
  if (p.stages != 0 && (rb.vec * sizeof(float) != 16 || p.stages < 2 || p.stages > 3 ||
                        p.stage_ns < 1 || p.stage_ns > 2))
    return cudaErrorInvalidValue;
  if (dry) return cudaSuccess;
  const size_t smem = red_smem_bytes(p, rb.vec, p.stages, p.stage_ns);
  cudaError_t e;
  if (p.cluster > 1) {
    return p.inner_kept
               ? launch_k_cluster(with_smem(k_reduce<OP, WHICH, 4, true, true>, smem), p.n_cta,
                                  kThreads, smem, s, p.cluster, p)
               : launch_k_cluster(with_smem(k_reduce<OP, WHICH, 4, false, true>, smem), p.n_cta,
                                  kThreads, smem, s, p.cluster, p);
  }
  if (p.inner_kept) {
    e = rb.vec == 4
            ? launch_k(with_smem(k_reduce<OP, WHICH, 4, true>, smem), p.n_cta, kThreads, smem, s, p)
            : launch_k(k_reduce<OP, WHICH, 1, true>, p.n_cta, kThreads, smem, s, p);
  } else {
    e = rb.vec == 4
            ? launch_k(with_smem(k_reduce<OP, WHICH, 4, false>, smem), p.n_cta, kThreads, smem, s, p)
            : launch_k(k_reduce<OP, WHICH, 1, false>, p.n_cta, kThreads, smem, s, p);
  }
  if (e != cudaSuccess || p.nslots <= 1) return e;
  return launch_combine_f32(rb.comb, s);
}

template <int OP>
cudaError_t launch_red_op(int which, const RedBuild& rb, cudaStream_t s, bool dry) {
  return which == 0 ? launch_red_t<OP, 0>(rb, s, dry) : launch_red_t<OP, 1>(rb, s, dry);
}

}  // namespace

cudaError_t launch_combine_f32(CombinePlan c, cudaStream_t s) {
  combine_vectorize(&c);
  const unsigned nblk = static_cast<unsigned>(combine_blocks(c));
  return c.vec == 4 ? launch_k(k_combine<float, 4>, nblk, kThreads, 0, s, c)
                    : launch_k(k_combine<float, 1>, nblk, kThreads, 0, s, c);
}

cudaError_t occupancy_red(int which, int* planned, int* actual) {
  // The largest dynamic shared memory a plan asks for: a full offset table
  // and the column-lane tree.
  const size_t smem = size_t(kMaxTileRows) * kMaxOperands * sizeof(int64_t) +
                      size_t(kThreads) * 4 * sizeof(float);
  switch (which) {
    case 0:
      *planned = kOccRedAddSub;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_reduce<OP_ADD, 1, 4, true>,
                                                           kThreads, smem);
    case 1:
      *planned = kOccRedAddSub;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_reduce<OP_SUB, 1, 4, false>,
                                                           kThreads, smem);
    case 2:
      *planned = kOccRedMulDiv;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_reduce<OP_MUL, 1, 4, true>,
                                                           kThreads, smem);
    case 3:
      *planned = kOccRedMulDiv;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_reduce<OP_DIV, 1, 4, false>,
                                                           kThreads, smem);
    case 4:
      *planned = kOccRedAddSub;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_reduce<OP_ADD, 2, 4, true>,
                                                           kThreads, smem);
    case 5:
      *planned = red_cl_occ(OP_ADD, true);
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_reduce<OP_ADD, 1, 4, true, true>, kThreads, smem);
    case 6:
      *planned = red_cl_occ(OP_SUB, false);
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_reduce<OP_SUB, 1, 4, false, true>, kThreads, smem);
    case 7:
      *planned = red_cl_occ(OP_MUL, true);
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_reduce<OP_MUL, 1, 4, true, true>, kThreads, smem);
    case 8:
      *planned = red_cl_occ(OP_DIV, false);
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_reduce<OP_DIV, 1, 4, false, true>, kThreads, smem);
    case 9:
      *planned = red_cl_occ(OP_ADD, true);
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          actual, k_reduce<OP_ADD, 2, 4, true, true>, kThreads, smem);
    case 10: {
      // Staged: c4's mask gradient (96 rows per CTA, three 16 KB batches).
      *planned = kOccRedAddSub;
      const size_t staged = size_t(96) * kMaxOperands * sizeof(int64_t) + 3 * kStageBatchBytes;
      const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(k_reduce<OP_ADD, 1, 4, true>));
      if (e != cudaSuccess) return e;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(actual, k_reduce<OP_ADD, 1, 4, true>,
                                                           kThreads, staged);
    }
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_reduce(int op, int which, const RedBuild& rb, cudaStream_t s, bool dry) {
  if (rb.es == 2) return launch_reduce_bf16(op, which, rb, s, dry);
  if (which == 2) return launch_red_t<OP_ADD, 2>(rb, s, dry);
  switch (op) {
    case OP_ADD: return launch_red_op<OP_ADD>(which, rb, s, dry);
    case OP_SUB: return launch_red_op<OP_SUB>(which, rb, s, dry);
    case OP_MUL: return launch_red_op<OP_MUL>(which, rb, s, dry);
    default: return launch_red_op<OP_DIV>(which, rb, s, dry);
  }
}

}  // namespace zr
