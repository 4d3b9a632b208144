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
// that beta are staged into shared memory by cp.async through a
// kSabStages-deep pipeline, so several tiles' loads are in flight while the
// previous one is summed and no load sits on the per-step critical path.
#pragma once

#include <cuda_runtime.h>
#include "zr_internal.h"
#include "zr_kernels.cuh"

namespace zr {

// The factor of b applied per element to grad_a's term is staged as a row
// of shared memory one step ahead: for div the row holds 1/b (so the per
// element work is one multiply), for mul it holds b.
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

template <int OP, int RPT>
__global__ void __launch_bounds__(kSabThreads, 1)
k_sab(const __grid_constant__ SabPlan p) {
  pdl_trigger();
  constexpr bool kUsesA = OP == OP_MUL || OP == OP_DIV;
  constexpr bool kUsesB = OP == OP_MUL || OP == OP_DIV;
  constexpr uint32_t kWarps = kSabThreads / 32;
  extern __shared__ float4 s_raw[];
  // Stage = tile [ta][ncol] followed by b's row [ncol] (converted in place
  // to the per-element factor one step before use).
  const uint32_t tile_floats = p.ta * p.ncol;
  const uint32_t stage_floats = tile_floats + p.ncol;
  const uint32_t ring_floats = (kWarps + 1) * p.ncol;  // [warps][ncol] + factors [ncol]
  float* s_stage = reinterpret_cast<float*>(s_raw);
  int64_t* s_row = reinterpret_cast<int64_t*>(s_stage + kSabStages * stage_floats);  // [ta][2]
  int64_t* s_beta = s_row + 2 * p.ta;                                                 // [n_beta][2]
  float* s_ring = reinterpret_cast<float*>(s_beta + 2 * p.n_beta);                    // [ring+1][...]

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
  const uint32_t n_steps = static_cast<uint32_t>(sab_start(p, cta + 1) - s0);
  const uint32_t nvc = p.nvc;  // power of two
  const uint32_t nvc_shift = __ffs(nvc) - 1;
  const uint32_t ncol_shift = nvc_shift + 2;
  const uint32_t lanes = kSabThreads >> nvc_shift;  // row lanes
  const uint32_t tx = tid & (nvc - 1);
  const uint32_t ty = tid >> nvc_shift;
  const uint32_t warp = tid >> 5, lane = tid & 31;
  const uint32_t R = p.ring;  // power of two

  // This thread's RPT 16-byte chunks of every tile: fixed rows and columns,
  // so their source offsets (within a tile) and destinations are fixed too.
  int64_t chunk_src[RPT];
  uint32_t chunk_dst[RPT];
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    const uint32_t id = tid + k * kSabThreads;
    const uint32_t row = id >> nvc_shift;
    const uint32_t c4 = id & (nvc - 1);
    chunk_src[k] = s_row[2 * row] + c4 * 4;
    chunk_dst[k] = row * p.ncol + c4 * 4;
  }
  pdl_wait();
  const uint32_t tile0 = fd_div(p.n_beta_div, static_cast<uint32_t>(s0));
  const uint32_t beta0 = static_cast<uint32_t>(s0) - tile0 * p.n_beta;
  auto g_base = [&](uint32_t tile) {
    int64_t ob[kMaxOperands];
    decomp_offsets(p.a_outer, tile, ob);
    return ob[0];
  };

  // Loads are issued in step order; (tile, beta) of the next one to issue.
  uint32_t iss_k = 0, iss_tile = tile0, iss_beta = beta0;
  int64_t iss_base = n_steps ? g_base(tile0) : 0;
  // Stage the next step's tile (and b's row) if in range; close one group.
  auto issue = [&](uint32_t stage) {
    if (iss_k < n_steps) {
      const float* src = p.g + iss_base + s_beta[2 * iss_beta];
      float* dst = s_stage + stage * stage_floats;
      if (kUsesB && tid < nvc)
        cp_async16(dst + tile_floats + tid * 4, p.b + s_beta[2 * iss_beta + 1] + tid * 4);
#pragma unroll
      for (int k = 0; k < RPT; ++k) cp_async16(dst + chunk_dst[k], src + chunk_src[k]);
      ++iss_k;
      if (++iss_beta == p.n_beta) {
        iss_beta = 0;
        ++iss_tile;
        if (iss_k < n_steps) iss_base = g_base(iss_tile);
      }
    }
    cp_async_commit();
  };
  // Turn a landed stage's b row into the per-element factor.
  auto convert_row = [&](uint32_t stage) {
    if (kUsesB && tid < p.ncol) {
      float* r = s_stage + stage * stage_floats + tile_floats;
      r[tid] = sab_row<OP>(r[tid]);
    }
  };
  // grad_b of `cnt` finished steps k0.. (ring entries rb0..): thread
  // (r, col) adds step k0+r's warp partials of column col in warp order,
  // scales by b's factor and stores to slot `tile` of the workspace.
  auto finish_b = [&](uint32_t k0, uint32_t cnt, uint32_t rb0) {
    const uint32_t r = tid >> ncol_shift, col = tid & (p.ncol - 1);
    if (r < cnt) {
      uint32_t rb = rb0 + r;
      if (rb > R) rb -= R + 1;
      const float* src = s_ring + rb * ring_floats + col;
      float v = src[0];
#pragma unroll
      for (uint32_t w = 1; w < kWarps; ++w) v = __fadd_rn(v, src[w * p.ncol]);
      const float rv = src[kWarps * p.ncol];
      const uint32_t step = static_cast<uint32_t>(s0) + k0 + r;
      const uint32_t tile = fd_div(p.n_beta_div, step);
      const uint32_t beta = step - tile * p.n_beta;
      const uint64_t jb = uint64_t(beta) * p.ncol + col;
      if (OP == OP_DIV) {
        // Unscaled partial; the tile-0 step (exactly one per beta) stores the
        // factor -1/b^2 after the slots, and the second pass multiplies each
        // total by it, so no partial can overflow on its own.
        p.ws_b[uint64_t(tile) * p.n_b + jb] = v;
        if (tile == 0) p.ws_b[uint64_t(p.n_tiles) * p.n_b + jb] = sab_scale<OP>(rv);
      } else {
        p.ws_b[uint64_t(tile) * p.n_b + jb] = __fmul_rn(v, sab_scale<OP>(rv));
      }
    }
  };

  for (int k = 0; k < kSabStages - 1; ++k) issue(k);
  cp_async_wait<kSabStages - 2>();
  __syncthreads();
  convert_row(0);

  // grad_a: per step a plain FMA into blk; every kSabFold steps (and when a
  // tile's partial is written) blk is added into the Kahan total acc.
  Kahan acc[RPT][4];
  float4 blk[RPT];
#pragma unroll
  for (int j = 0; j < RPT; ++j) {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i].init();
    blk[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float4 areg[RPT];
#pragma unroll
  for (int j = 0; j < RPT; ++j) areg[j] = make_float4(1.f, 1.f, 1.f, 1.f);
  uint32_t tile = tile0, beta = beta0;
  uint32_t sc = 0;       // stage of step k
  uint32_t wr = 0;       // ring entry of step k (k mod (R + 1))
  uint32_t nfold = 0;    // steps in blk

  for (uint32_t k = 0; k < n_steps; ++k) {
    // Steps k and k+1 have landed (for this thread's copies); the barrier
    // makes every thread's copies visible and frees stage (k-1).
    cp_async_wait<kSabStages - 3>();
    __syncthreads();
    const uint32_t s_next = sc + 1 == kSabStages ? 0 : sc + 1;
    if (k + 1 < n_steps) convert_row(s_next);
    // Ring entries of steps k-R .. k-1 are complete (k-R sits at wr+1).
    if (k != 0 && (k & (R - 1)) == 0) finish_b(k - R, R, wr == R ? 0 : wr + 1);
    issue(sc == 0 ? kSabStages - 1 : sc - 1);

    if (kUsesA && (k == 0 || beta == 0)) {
      int64_t ob[kMaxOperands];
      decomp_offsets(p.a_outer, tile, ob);
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        const uint32_t row = ty + j * lanes;
        areg[j] = __ldg(reinterpret_cast<const float4*>(p.a + ob[1] + s_row[2 * row + 1] + tx * 4));
      }
    }
    const float* st = s_stage + sc * stage_floats;
    float* ring = s_ring + wr * ring_floats;
    float4 ca = make_float4(1.f, 1.f, 1.f, 1.f);
    if (kUsesB) {
      ca = *reinterpret_cast<const float4*>(st + tile_floats + tx * 4);
      if (tid < p.ncol) ring[kWarps * p.ncol + tid] = st[tile_floats + tid];
    }

    float4 sb = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < RPT; ++j) {
      const uint32_t row = ty + j * lanes;
      const float4 g4 = *reinterpret_cast<const float4*>(st + row * p.ncol + tx * 4);
      if (OP == OP_ADD || OP == OP_SUB) {
        blk[j].x = __fadd_rn(blk[j].x, g4.x); blk[j].y = __fadd_rn(blk[j].y, g4.y);
        blk[j].z = __fadd_rn(blk[j].z, g4.z); blk[j].w = __fadd_rn(blk[j].w, g4.w);
        sb.x = __fadd_rn(sb.x, g4.x); sb.y = __fadd_rn(sb.y, g4.y);
        sb.z = __fadd_rn(sb.z, g4.z); sb.w = __fadd_rn(sb.w, g4.w);
      } else {
        blk[j].x = __fmaf_rn(g4.x, ca.x, blk[j].x); blk[j].y = __fmaf_rn(g4.y, ca.y, blk[j].y);
        blk[j].z = __fmaf_rn(g4.z, ca.z, blk[j].z); blk[j].w = __fmaf_rn(g4.w, ca.w, blk[j].w);
        sb.x = __fmaf_rn(g4.x, areg[j].x, sb.x);
        sb.y = __fmaf_rn(g4.y, areg[j].y, sb.y);
        sb.z = __fmaf_rn(g4.z, areg[j].z, sb.z);
        sb.w = __fmaf_rn(g4.w, areg[j].w, sb.w);
      }
    }
    // Lanes of a warp that share tx hold different rows: butterfly over them.
    for (uint32_t off = nvc; off < 32; off <<= 1) {
      sb.x = __fadd_rn(sb.x, __shfl_xor_sync(0xffffffffu, sb.x, off));
      sb.y = __fadd_rn(sb.y, __shfl_xor_sync(0xffffffffu, sb.y, off));
      sb.z = __fadd_rn(sb.z, __shfl_xor_sync(0xffffffffu, sb.z, off));
      sb.w = __fadd_rn(sb.w, __shfl_xor_sync(0xffffffffu, sb.w, off));
    }
    if (lane < nvc) *reinterpret_cast<float4*>(ring + warp * p.ncol + tx * 4) = sb;

    // Leaving this tile (its last beta, or the end of this CTA's range):
    // write grad_a's partial to this CTA's slot for the tile.
    const bool tile_done = beta == p.n_beta - 1;
    const bool leave = tile_done || k + 1 == n_steps;
    if (++nfold == kSabFold || leave) {
#pragma unroll
      for (int j = 0; j < RPT; ++j) {
        acc[j][0].add(blk[j].x); acc[j][1].add(blk[j].y);
        acc[j][2].add(blk[j].z); acc[j][3].add(blk[j].w);
        blk[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      nfold = 0;
    }
    if (leave) {
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
    if (tile_done) {
      beta = 0;
      ++tile;
    } else {
      ++beta;
    }
    sc = s_next;
    wr = wr == R ? 0 : wr + 1;
  }
  cp_async_wait<0>();
  __syncthreads();
  // Steps left in the ring: from the last multiple of R below n_steps.
  if (n_steps > 0) {
    const uint32_t k0 = ((n_steps - 1) / R) * R;
    finish_b(k0, n_steps - k0, k0 % (R + 1));
  }
}

}  // namespace zr
