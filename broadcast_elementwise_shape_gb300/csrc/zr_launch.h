// zr_launch.h — kernel launchers (one translation unit per kernel family so
// the library builds in parallel).
#pragma once

#include <cuda_runtime.h>

#include <mutex>
#include <utility>
#include <vector>

#include "zr_plan.h"

namespace zr {

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the kernel before it in the stream is still running.  Every kernel
// of this library calls pdl_wait() (griddepcontrol.wait, which returns once
// the grids before it have completed and their writes are visible) before
// its first global memory access, so only launch latency and parameter-only
// setup overlap the previous kernel, never a memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                            cudaStream_t s, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The same launch with the grid split into thread-block clusters of
// `cluster` CTAs along x.  Sizes above 8 are non-portable and need the
// kernel's opt-in attribute, which is set on first use.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k_cluster(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                                    size_t smem, cudaStream_t s, unsigned cluster,
                                    const Args&... args) {
  if (cluster > 8) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Kernels whose dynamic shared memory may exceed the default 48 KB limit:
// raise_smem_limit sets the kernel's limit to the most a CTA may use, once
// per kernel and device (remembered in a small table under a lock).
inline cudaError_t raise_smem_limit(const void* kernel) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& d : done)
    if (d.first == kernel && d.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e == cudaSuccess) done.emplace_back(kernel, dev);
  return e;
}
// The kernel itself when `smem` bytes are allowed for it, null otherwise (the
// launch then fails with an error instead of running short of memory).
template <typename... KArgs>
inline auto with_smem(void (*kernel)(KArgs...), size_t smem) -> void (*)(KArgs...) {
  if (smem <= 48 * 1024) return kernel;
  return raise_smem_limit(reinterpret_cast<const void*>(kernel)) == cudaSuccess ? kernel : nullptr;
}

// Every launcher first checks that the plan provides each operand its kernel
// dereferences (cudaErrorInvalidValue otherwise); with dry == true it stops
// there and launches nothing.
cudaError_t launch_fwd(int op, const EwBuild& eb, cudaStream_t s, bool dry = false);
// Split forward (each outer dim varies in exactly one input).
cudaError_t launch_fwd_sabf(int op, int rpt, const SabFPlan& sp, cudaStream_t s, bool dry = false);
// Forward with a transposed input (shared-memory tile transpose).
cudaError_t launch_fwd_tr(int op, const TrPlan& tp, cudaStream_t s, bool dry = false);
// want: bit 0 grad_a, bit 1 grad_b (no reduction).
cudaError_t launch_bwd_direct(int op, int want, const EwBuild& eb, cudaStream_t s, bool dry = false);
cudaError_t launch_copy(const EwBuild& eb, cudaStream_t s, bool dry = false);
// Unary ops (UnaryCode): forward (slot 0 = x) and backward (slot 0 = grad_out,
// slot 1 = x); eb.plan.alpha is scale's factor.
cudaError_t launch_unary_fwd(int uop, const EwBuild& eb, cudaStream_t s, bool dry = false);
cudaError_t launch_unary_bwd(int uop, const EwBuild& eb, cudaStream_t s, bool dry = false);
// which: 0 = grad_a, 1 = grad_b, 2 = sum-to-shape.  Launches the reduction
// pass and, when it writes partials, the combine pass.
cudaError_t launch_reduce(int op, int which, const RedBuild& rb, cudaStream_t s, bool dry = false);

// Resident CTAs per SM of one representative instantiation per kernel
// family (the 16-byte-vector variants the workloads run), as the planner
// assumes (*planned) and as the runtime reports for the current device
// (*actual).  ew: 0 fwd add, 1 fwd div, 2 bwd div (both gradients), 3 copy,
// 4 GeLU forward, 5 GeLU backward, 6 flat fwd add, 7 flat GeLU forward;
// bf16: 0 flat 8-wide GeLU forward;
// red: 0 add inner kept, 1 sub inner reduced, 2 mul inner kept, 3 div inner
// reduced, 4 sum-to-shape; 5..9 the same five as cluster variants; 10 add
// inner kept with a three-batch staging ring; other: 0 k_sabf (8 rows per
// thread), 1 k_transpose.
cudaError_t occupancy_ew(int which, int* planned, int* actual);
cudaError_t occupancy_bf16(int which, int* planned, int* actual);
cudaError_t occupancy_red(int which, int* planned, int* actual);
cudaError_t occupancy_other(int which, int* planned, int* actual);

// bfloat16 storage (plans with es == 2): the float launchers above hand
// those plans to these.
cudaError_t launch_fwd_bf16(int op, const EwBuild& eb, cudaStream_t s, bool dry);
cudaError_t launch_bwd_direct_bf16(int op, int want, const EwBuild& eb, cudaStream_t s, bool dry);
cudaError_t launch_copy_bf16(const EwBuild& eb, cudaStream_t s, bool dry);
// Second pass of a reduction whose partial pointer is set: 4 outputs per
// thread where combine_vectorize allows it.
cudaError_t launch_combine_f32(CombinePlan c, cudaStream_t s);
cudaError_t launch_combine_bf16(CombinePlan c, cudaStream_t s);
cudaError_t launch_unary_fwd_bf16(int uop, const EwBuild& eb, cudaStream_t s, bool dry);
cudaError_t launch_unary_bwd_bf16(int uop, const EwBuild& eb, cudaStream_t s, bool dry);
// Test kernel: the two bfloat16 divisions against the IEEE divide over all
// bfloat16 pairs.
cudaError_t launch_div_short_check(unsigned long long* out, cudaStream_t s);
cudaError_t launch_reduce_bf16(int op, int which, const RedBuild& rb, cudaStream_t s, bool dry);

// Two-op chains out = (a op1 b) op2 c: the forward (slots 0..2 = a, b, c)
// and the fused one-pass backward with its second passes.
// c_one: c has one element (read once per thread, 4 CTAs per SM).
cudaError_t launch_chain_fwd(int op1, int op2, bool c_one, const EwBuild& eb, cudaStream_t s,
                             bool dry = false);
cudaError_t launch_chain_bwd(int op1, int op2, const ChainBuild& cb, cudaStream_t s, bool dry = false);
// 0: chain forward (mul, add); 1: fused backward (mul, add), c shaped like b;
// 2: fused backward (add, div), c one element; 3: chain forward (add, div), c
// one element.
cudaError_t occupancy_chain(int which, int* planned, int* actual);

// Fused backward with both gradients reduced: the k_sab pass, then one
// combine pass per gradient.  sb.plan.ws_a / ws_b must be set.
cudaError_t launch_sab(int op, const SabBuild& sb, cudaStream_t s, bool dry = false);

}  // namespace zr
