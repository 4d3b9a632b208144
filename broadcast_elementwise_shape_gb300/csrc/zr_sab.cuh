// zr_sab.cuh — fused backward for a broadcast where BOTH gradients are
// reduced (every output dim except the innermost is kept by exactly one
// input), e.g. a [4,1,8,1,16,1,32,64] op b [1,6,1,12,1,10,1,64].
//
// Zero book, Operator page, section 广播: repetition in the forward pass is
// summation in the backward pass; here each grad_out element is summed into
// one element of grad_a AND one of grad_b, and both sums are formed in one
// read of grad_out.  With alpha = position along a's own dims and beta along
// b's, grad_out is g[alpha, beta, col] and
//   grad_a[alpha, col] = sum_beta  g * ca(beta, col)
//   grad_b[beta, col]  = sb(beta, col) * sum_alpha g * cb(alpha, col)
// where (ca, cb, sb) = (1, 1, 1) add, (1, 1, -1) sub, (b, a, 1) mul,
// (1/b, a, -1/b^2) div — the local terms of add (GPU page, section OpAdd),
// mul (Operator page, section 逐元素算子) and the calculus rules for sub/div,
// with b's factor taken out of the alpha sum.
//
// Persistent grid; each CTA walks a contiguous range of steps (tile, beta).
// A step's tile (ta rows x ncol floats, typically 32 KB) is staged into
// shared memory by cp.async through a kSabStages-deep pipeline, so several
// tiles' loads are in flight while the previous one is summed.
#pragma once

#include <cuda_runtime.h>
#include "zr_internal.h"
#include "zr_kernels.cuh"

namespace zr {

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// b's factor in grad_a's term, per lane.
template <int OP>
__device__ __forceinline__ float sab_ca(float bv) {
  if (OP == OP_MUL) return bv;
  if (OP == OP_DIV) return __frcp_rn(bv);
  return 1.0f;
}
// b's factor applied to grad_b's alpha sum.
template <int OP>
__device__ __forceinline__ float sab_sb(float bv) {
  if (OP == OP_SUB) return -1.0f;
  if (OP == OP_DIV) {
    const float r = __frcp_rn(bv);
    return -__fmul_rn(r, r);
  }
  return 1.0f;
}

template <int OP, int RPT>
__global__ void __launch_bounds__(kThreads, 1)
k_sab(const __grid_constant__ SabPlan p) {
  constexpr bool kUsesA = OP == OP_MUL || OP == OP_DIV;
  constexpr bool kUsesB = OP == OP_MUL || OP == OP_DIV;
  extern __shared__ float4 s_raw[];
  const uint32_t tile_floats = p.ta * p.ncol;
  float* s_stage = reinterpret_cast<float*>(s_raw);
  int64_t* s_row = reinterpret_cast<int64_t*>(s_stage + kSabStages * tile_floats);  // [ta][2]
  int64_t* s_beta = s_row + 2 * p.ta;                                                // [n_beta][2]
  float* s_sb = reinterpret_cast<float*>(s_beta + 2 * p.n_beta);                     // [2][8][ncol]

  const uint32_t tid = threadIdx.x;
  for (uint32_t i = tid; i < p.ta; i += blockDim.x) {
    int64_t off[kMaxOperands];
    decomp_offsets(p.a_inner, i, off);
    s_row[2 * i] = off[0];
    s_row[2 * i + 1] = off[1];
  }
  for (uint32_t i = tid; i < p.n_beta; i += blockDim.x) {
    int64_t off[kMaxOperands];
    decomp_offsets(p.beta, i, off);
    s_beta[2 * i] = off[0];
    s_beta[2 * i + 1] = off[2];
  }
  __syncthreads();

  const uint32_t cta = blockIdx.x;
  const uint64_t s0 = sab_start(p, cta);
  const uint64_t s1 = sab_start(p, cta + 1);
  const uint32_t nvc = p.nvc;  // power of two
  const uint32_t nvc_shift = __ffs(nvc) - 1;
  const uint32_t lanes = kThreads >> nvc_shift;  // row lanes
  const uint32_t tx = tid & (nvc - 1);
  const uint32_t ty = tid >> nvc_shift;
  const uint32_t warp = tid >> 5, lane = tid & 31;

  // Stage the tile of step `step` (if in range) and close one copy group.
  auto issue = [&](uint64_t step, uint32_t stage) {
    if (step < s1) {
      const uint32_t tile = fd_div(p.n_beta_div, static_cast<uint32_t>(step));
      const uint32_t beta = static_cast<uint32_t>(step) - tile * p.n_beta;
      int64_t ob[kMaxOperands];
      decomp_offsets(p.a_outer, tile, ob);
      const float* src = p.g + ob[0] + s_beta[2 * beta];
      float* dst = s_stage + stage * tile_floats;
#pragma unroll
      for (int k = 0; k < RPT; ++k) {
        const uint32_t id = tid + k * kThreads;
        const uint32_t row = id >> nvc_shift;
        const uint32_t c4 = id & (nvc - 1);
        cp_async16(dst + row * p.ncol + c4 * 4, src + s_row[2 * row] + c4 * 4);
      }
    }
    cp_async_commit();
  };

  // grad_b of one finished step: add the 8 warps' partials in warp order,
  // apply b's factor, store to slot `tile` of the workspace.
  auto finish_b = [&](uint64_t step, uint32_t buf, float4 bv) {
    if (tid < nvc) {
      const uint32_t tile = fd_div(p.n_beta_div, static_cast<uint32_t>(step));
      const uint32_t beta = static_cast<uint32_t>(step) - tile * p.n_beta;
      const float* src = s_sb + buf * 8 * p.ncol + tid * 4;
      float4 v = *reinterpret_cast<const float4*>(src);
      for (int w = 1; w < 8; ++w) {
        const float4 u = *reinterpret_cast<const float4*>(src + w * p.ncol);
        v.x = __fadd_rn(v.x, u.x); v.y = __fadd_rn(v.y, u.y);
        v.z = __fadd_rn(v.z, u.z); v.w = __fadd_rn(v.w, u.w);
      }
      v.x = __fmul_rn(v.x, sab_sb<OP>(bv.x)); v.y = __fmul_rn(v.y, sab_sb<OP>(bv.y));
      v.z = __fmul_rn(v.z, sab_sb<OP>(bv.z)); v.w = __fmul_rn(v.w, sab_sb<OP>(bv.w));
      float* dst = p.ws_b + uint64_t(tile) * p.n_b + uint64_t(beta) * p.ncol + tid * 4;
      *reinterpret_cast<float4*>(dst) = v;
    }
  };

  for (int k = 0; k < kSabStages - 1; ++k) issue(s0 + k, k);

  Kahan acc[RPT][4];
#pragma unroll
  for (int j = 0; j < RPT; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i].init();
  float4 areg[RPT];
#pragma unroll
  for (int j = 0; j < RPT; ++j) areg[j] = make_float4(1.f, 1.f, 1.f, 1.f);
  uint32_t cur_tile = 0xffffffffu;
  float4 bcur = make_float4(1.f, 1.f, 1.f, 1.f), bprev = bcur;

  for (uint64_t step = s0; step < s1; ++step) {
    const uint32_t k = static_cast<uint32_t>(step - s0);
    cp_async_wait<kSabStages - 2>();
    __syncthreads();
    if (k > 0) finish_b(step - 1, (k - 1) & 1, bprev);
    issue(step + kSabStages - 1, (k + kSabStages - 1) % kSabStages);

    const uint32_t tile = fd_div(p.n_beta_div, static_cast<uint32_t>(step));
    const uint32_t beta = static_cast<uint32_t>(step) - tile * p.n_beta;
    if (kUsesA && tile != cur_tile) {
      int64_t ob[kMaxOperands];
      decomp_offsets(p.a_outer, tile, ob);
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        const uint32_t row = ty + j * lanes;
        areg[j] = __ldg(reinterpret_cast<const float4*>(p.a + ob[1] + s_row[2 * row + 1] + tx * 4));
      }
    }
    cur_tile = tile;
    if (kUsesB) bcur = __ldg(reinterpret_cast<const float4*>(p.b + s_beta[2 * beta + 1] + tx * 4));
    const float4 ca = make_float4(sab_ca<OP>(bcur.x), sab_ca<OP>(bcur.y), sab_ca<OP>(bcur.z),
                                  sab_ca<OP>(bcur.w));

    const float* st = s_stage + (k % kSabStages) * tile_floats;
    float4 sb = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const uint32_t row = ty + j * lanes;
      const float4 g4 = *reinterpret_cast<const float4*>(st + row * p.ncol + tx * 4);
      if (OP == OP_ADD || OP == OP_SUB) {
        acc[j][0].add(g4.x); acc[j][1].add(g4.y); acc[j][2].add(g4.z); acc[j][3].add(g4.w);
        sb.x = __fadd_rn(sb.x, g4.x); sb.y = __fadd_rn(sb.y, g4.y);
        sb.z = __fadd_rn(sb.z, g4.z); sb.w = __fadd_rn(sb.w, g4.w);
      } else {
        acc[j][0].add(__fmul_rn(g4.x, ca.x)); acc[j][1].add(__fmul_rn(g4.y, ca.y));
        acc[j][2].add(__fmul_rn(g4.z, ca.z)); acc[j][3].add(__fmul_rn(g4.w, ca.w));
        sb.x = __fadd_rn(sb.x, __fmul_rn(g4.x, areg[j].x));
        sb.y = __fadd_rn(sb.y, __fmul_rn(g4.y, areg[j].y));
        sb.z = __fadd_rn(sb.z, __fmul_rn(g4.z, areg[j].z));
        sb.w = __fadd_rn(sb.w, __fmul_rn(g4.w, areg[j].w));
      }
    }
    // Lanes of a warp that share tx hold different rows: butterfly over them.
    for (uint32_t off = nvc; off < 32; off <<= 1) {
      sb.x = __fadd_rn(sb.x, __shfl_xor_sync(0xffffffffu, sb.x, off));
      sb.y = __fadd_rn(sb.y, __shfl_xor_sync(0xffffffffu, sb.y, off));
      sb.z = __fadd_rn(sb.z, __shfl_xor_sync(0xffffffffu, sb.z, off));
      sb.w = __fadd_rn(sb.w, __shfl_xor_sync(0xffffffffu, sb.w, off));
    }
    if (lane < nvc)
      *reinterpret_cast<float4*>(s_sb + (k & 1) * 8 * p.ncol + warp * p.ncol + tx * 4) = sb;

    // Leaving this tile (its last beta, or the end of this CTA's range):
    // write grad_a's partial to this CTA's slot for the tile.
    const bool tile_done = beta == p.n_beta - 1;
    if (tile_done || step == s1 - 1) {
      const uint32_t slot = cta - sab_owner(p, uint64_t(tile) * p.n_beta);
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        const uint32_t row = ty + j * lanes;
        const uint64_t x = (uint64_t(tile) * p.ta + row) * p.ncol + tx * 4;
        const float4 v = make_float4(acc[j][0].s, acc[j][1].s, acc[j][2].s, acc[j][3].s);
        *reinterpret_cast<float4*>(p.ws_a + uint64_t(slot) * p.n_a + x) = v;
        if (tile_done) {
          // Slots no CTA reaches for this tile hold zeros.
          for (uint32_t s = slot + 1; s < p.slots_a; ++s)
            *reinterpret_cast<float4*>(p.ws_a + uint64_t(s) * p.n_a + x) =
                make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[j][i].init();
      }
    }
    bprev = bcur;
  }
  cp_async_wait<0>();
  __syncthreads();
  if (s1 > s0) finish_b(s1 - 1, static_cast<uint32_t>(s1 - s0 - 1) & 1, bprev);
}

}  // namespace zr
