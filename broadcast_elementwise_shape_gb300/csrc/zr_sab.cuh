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
// (each product enters its sum through an FMA, so it is never rounded on
// its own)
// where (ca, cb, sb) = (1, 1, 1) add, (1, 1, -1) sub, (b, a, 1) mul,
// (1/b, a, -1/b^2) div — the local terms of add (GPU page, section OpAdd),
// mul (Operator page, section 逐元素算子) and the calculus rules for sub/div,
// with b's factor taken out of the alpha sum.
//
// Persistent grid; each CTA walks a contiguous range of steps (tile, beta).
// A step's tile (ta rows x ncol floats, typically 32 KB) and b's row for
// that beta are staged into shared memory by TMA bulk copies (one per run of
// rows contiguous in g) through a kSabStages-deep ring of stage barriers,
// so several tiles' loads are in flight while the previous one is summed and
// no load sits on the per-step critical path.
#pragma once

#include <cuda_runtime.h>
#include "zr_internal.h"
#include "zr_kernels.cuh"

namespace zr {

// ---- TMA bulk copies and stage barriers (inline PTX, sm_90 and later) ----

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
// Make barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// Order this thread's earlier generic shared-memory accesses before later
// bulk copies into the same memory.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  uint64_t state;
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;\n"
               : "=l"(state) : "r"(smem_addr(bar)), "r"(bytes) : "memory");
  (void)state;
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return done != 0;
}
// Bounded wait for the phase of parity `parity` to complete.  Returns false
// if it did not within the limit (each try_wait may itself suspend a while),
// so a broken pipeline ends the kernel instead of hanging the GPU.
constexpr uint32_t kWaitLimit = 1u << 22;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// The factor of b applied per element to grad_a's term, staged as a row of
// shared memory one step ahead: 1/b for div, b for mul.
template <int OP>
__device__ __forceinline__ float sab_row(float bv) {
  return OP == OP_DIV ? __frcp_rn(bv) : bv;
}
// Factor applied to grad_b's alpha sum, from the staged row value.
template <int OP>
__device__ __forceinline__ float sab_scale(float rv) {
  if (OP == OP_SUB) return -1.0f;
  if (OP == OP_DIV) return -__fmul_rn(rv, rv);
  return 1.0f;
}

// grad_a accumulation: each thread adds one term per step per element into
// a plain register sum (an FMA), and every kSabFold steps folds those sums
// into Kahan totals kept in shared memory; error <= (kSabFold + 2) u
// sum|terms|, however many steps a thread covers.
template <int RPT>
__device__ __forceinline__ void sab_fold(float4 (&blk)[RPT], float* ks, float* kc, uint32_t tid) {
#pragma unroll
  for (int j = 0; j < RPT; ++j) {
    const float v[4] = {blk[j].x, blk[j].y, blk[j].z, blk[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t idx = (j * 4 + i) * kSabThreads + tid;
      const float c = kc[idx], s = ks[idx];
      const float y = __fsub_rn(v[i], c);
      const float t = __fadd_rn(s, y);
      kc[idx] = __fsub_rn(__fsub_rn(t, s), y);
      ks[idx] = t;
    }
    blk[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <int OP, int RPT>
__global__ void __launch_bounds__(kSabThreads, 1)
k_sab(const __grid_constant__ SabPlan p) {
  constexpr bool kUsesA = OP == OP_MUL || OP == OP_DIV;
  constexpr bool kUsesB = OP == OP_MUL || OP == OP_DIV;
  constexpr uint32_t kWarps = kSabThreads / 32;
  extern __shared__ float4 s_raw[];
  // Stage = tile [ta][ncol] followed by b's row [ncol] (converted in place
  // to the per-element factor one step before use).
  const uint32_t tile_floats = p.ta * p.ncol;
  const uint32_t stage_floats = tile_floats + p.ncol;
  float* s_stage = reinterpret_cast<float*>(s_raw);
  float* s_ks = s_stage + kSabStages * stage_floats;               // [RPT*4][threads]
  float* s_kc = s_ks + RPT * 4 * kSabThreads;                      // [RPT*4][threads]
  int64_t* s_row = reinterpret_cast<int64_t*>(s_kc + RPT * 4 * kSabThreads);  // [ta][2]
  int64_t* s_beta = s_row + 2 * p.ta;                                         // [n_beta][2]
  float* s_sb = reinterpret_cast<float*>(s_beta + 2 * p.n_beta);              // [2][warps][ncol]
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_sb + 2 * kWarps * p.ncol);  // [stages]
  __shared__ int s_abort;

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
  for (uint32_t i = tid; i < RPT * 4 * kSabThreads; i += blockDim.x) {
    s_ks[i] = 0.f;
    s_kc[i] = 0.f;
  }
  if (tid == 0) {
    for (int st = 0; st < kSabStages; ++st) mbar_init(&s_bar[st], 1);
    mbar_init_fence();
    s_abort = 0;
  }
  __syncthreads();

  const uint32_t cta = blockIdx.x;
  const uint64_t s0 = sab_start(p, cta);
  const uint64_t s1 = sab_start(p, cta + 1);
  const uint32_t nvc = p.nvc;  // power of two
  const uint32_t nvc_shift = __ffs(nvc) - 1;
  const uint32_t lanes = kSabThreads >> nvc_shift;  // row lanes
  const uint32_t tx = tid & (nvc - 1);
  const uint32_t ty = tid >> nvc_shift;
  const uint32_t warp = tid >> 5, lane = tid & 31;
  const uint32_t run_bytes = p.run_rows * p.ncol * 4;
  const uint32_t n_runs = p.ta / p.run_rows;
  const uint32_t step_bytes = tile_floats * 4 + (kUsesB ? p.ncol * 4 : 0);

  // Warp 0 stages step `step` into `stage`: lane 0 arms the stage barrier
  // with the byte count, then the lanes issue one bulk copy per row run and
  // one for b's row.
  uint32_t iss_tile = 0xffffffffu;
  int64_t iss_base = 0;
  auto issue = [&](uint64_t step, uint32_t stage) {
    if (warp != 0 || step >= s1) return;
    const uint32_t tile = fd_div(p.n_beta_div, static_cast<uint32_t>(step));
    const uint32_t beta = static_cast<uint32_t>(step) - tile * p.n_beta;
    if (tile != iss_tile) {
      int64_t ob[kMaxOperands];
      decomp_offsets(p.a_outer, tile, ob);
      iss_tile = tile;
      iss_base = ob[0];
    }
    const float* src = p.g + iss_base + s_beta[2 * beta];
    float* dst = s_stage + stage * stage_floats;
    if (lane == 0) {
      fence_proxy_async();
      mbar_arrive_expect_tx(&s_bar[stage], step_bytes);
    }
    __syncwarp();
    for (uint32_t r = lane; r < n_runs; r += 32)
      bulk_g2s(dst + r * p.run_rows * p.ncol, src + s_row[2 * r * p.run_rows], run_bytes, &s_bar[stage]);
    if (kUsesB && lane == 0)
      bulk_g2s(dst + tile_floats, p.b + s_beta[2 * beta + 1], p.ncol * 4, &s_bar[stage]);
  };
  auto parity_of = [&](uint32_t k) { return (k / kSabStages) & 1u; };
  // Turn a landed stage's b row into the per-element factor.
  auto convert_row = [&](uint32_t stage) {
    if (kUsesB && tid < p.ncol) {
      float* r = s_stage + stage * stage_floats + tile_floats;
      r[tid] = sab_row<OP>(r[tid]);
    }
  };
  // grad_b of a finished step: per column, the warps' partials in warp order,
  // times b's factor; stored to slot `tile` of the workspace.
  auto finish_b = [&](uint64_t step, uint32_t buf, float rv) {
    if (tid < p.ncol) {
      const uint32_t tile = fd_div(p.n_beta_div, static_cast<uint32_t>(step));
      const uint32_t beta = static_cast<uint32_t>(step) - tile * p.n_beta;
      const float* src = s_sb + buf * kWarps * p.ncol + tid;
      float v = src[0];
#pragma unroll
      for (uint32_t w = 1; w < kWarps; ++w) v = __fadd_rn(v, src[w * p.ncol]);
      p.ws_b[uint64_t(tile) * p.n_b + uint64_t(beta) * p.ncol + tid] = __fmul_rn(v, sab_scale<OP>(rv));
    }
  };

  for (uint32_t k = 0; k + 1 < kSabStages; ++k) issue(s0 + k, k);
  // Step 0's b row must be converted before anyone computes step 0.
  if (kUsesB && tid < p.ncol && s0 < s1) {
    if (mbar_wait(&s_bar[0], 0)) convert_row(0);
    else s_abort = 1;
  }

  float4 blk[RPT];
#pragma unroll
  for (int j = 0; j < RPT; ++j) blk[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 areg[RPT];
#pragma unroll
  for (int j = 0; j < RPT; ++j) areg[j] = make_float4(1.f, 1.f, 1.f, 1.f);
  uint32_t cur_tile = 0xffffffffu;
  uint32_t since_fold = 0;
  float rprev = 1.0f;  // factor of column tid at the previous step (tid < ncol)
  uint32_t k = 0;

  for (uint64_t step = s0; step < s1; ++step, ++k) {
    // Everyone is done with step k-1: its stage may be refilled and its
    // grad_b partials summed.
    __syncthreads();
    if (s_abort) break;
    issue(step + kSabStages - 1, (k + kSabStages - 1) % kSabStages);
    if (k > 0) finish_b(step - 1, (k - 1) & 1, rprev);
    if (kUsesB && tid < p.ncol && step + 1 < s1) {
      // Convert step k+1's b row now; it is read after the next barrier.
      if (mbar_wait(&s_bar[(k + 1) % kSabStages], parity_of(k + 1))) convert_row((k + 1) % kSabStages);
      else s_abort = 1;
    }
    if (!mbar_wait(&s_bar[k % kSabStages], parity_of(k))) {
      s_abort = 1;
      continue;
    }

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
    const float* st = s_stage + (k % kSabStages) * stage_floats;
    float4 ca = make_float4(1.f, 1.f, 1.f, 1.f);
    if (kUsesB) {
      ca = *reinterpret_cast<const float4*>(st + tile_floats + tx * 4);
      if (tid < p.ncol) rprev = st[tile_floats + tid];
    }

    float4 sb = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const uint32_t row = ty + j * lanes;
      const float4 g4 = *reinterpret_cast<const float4*>(st + row * p.ncol + tx * 4);
      blk[j].x = __fmaf_rn(g4.x, ca.x, blk[j].x);
      blk[j].y = __fmaf_rn(g4.y, ca.y, blk[j].y);
      blk[j].z = __fmaf_rn(g4.z, ca.z, blk[j].z);
      blk[j].w = __fmaf_rn(g4.w, ca.w, blk[j].w);
      if (kUsesA) {
        sb.x = __fmaf_rn(g4.x, areg[j].x, sb.x);
        sb.y = __fmaf_rn(g4.y, areg[j].y, sb.y);
        sb.z = __fmaf_rn(g4.z, areg[j].z, sb.z);
        sb.w = __fmaf_rn(g4.w, areg[j].w, sb.w);
      } else {
        sb.x = __fadd_rn(sb.x, g4.x); sb.y = __fadd_rn(sb.y, g4.y);
        sb.z = __fadd_rn(sb.z, g4.z); sb.w = __fadd_rn(sb.w, g4.w);
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
      *reinterpret_cast<float4*>(s_sb + (k & 1) * kWarps * p.ncol + warp * p.ncol + tx * 4) = sb;

    // Leaving this tile (its last beta, or the end of this CTA's range):
    // fold, then write grad_a's partial to this CTA's slot for the tile.
    const bool tile_done = beta == p.n_beta - 1;
    const bool leave = tile_done || step == s1 - 1;
    if (++since_fold == kSabFold || leave) {
      sab_fold<RPT>(blk, s_ks, s_kc, tid);
      since_fold = 0;
    }
    if (leave) {
      const uint32_t slot = cta - sab_owner(p, uint64_t(tile) * p.n_beta);
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        const uint32_t row = ty + j * lanes;
        const uint64_t x = (uint64_t(tile) * p.ta + row) * p.ncol + tx * 4;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t idx = (j * 4 + i) * kSabThreads + tid;
          v[i] = s_ks[idx];
          s_ks[idx] = 0.f;
          s_kc[idx] = 0.f;
        }
        *reinterpret_cast<float4*>(p.ws_a + uint64_t(slot) * p.n_a + x) = make_float4(v[0], v[1], v[2], v[3]);
        if (tile_done) {
          // Slots no CTA reaches for this tile hold zeros.
          for (uint32_t s = slot + 1; s < p.slots_a; ++s)
            *reinterpret_cast<float4*>(p.ws_a + uint64_t(s) * p.n_a + x) =
                make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
  __syncthreads();
  if (s_abort) {
    // Record the failure, and let every copy this CTA issued land before
    // its shared memory is released (each wait bounded again).
    if (tid == 0) {
      *p.status = 1;
      const uint64_t issued_end = s0 + k + kSabStages - 1 < s1 ? s0 + k + kSabStages - 1 : s1;
      for (uint64_t st = s0 + k; st < issued_end; ++st) {
        const uint32_t kk = static_cast<uint32_t>(st - s0);
        mbar_wait(&s_bar[kk % kSabStages], parity_of(kk));
      }
    }
    return;
  }
  if (s1 > s0) finish_b(s1 - 1, static_cast<uint32_t>(s1 - s0 - 1) & 1, rprev);
}

}  // namespace zr
