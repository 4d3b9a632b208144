// zr_chain.cuh — fused backward of a two-op chain out = (a op1 b) op2 c in
// one pass over grad_out (sm_103a).
//
// The Zero book's Operator page, section 融合 (fusion), fuses small
// operators so that one kernel launch and one pass over memory replace
// several, without changing the mathematics.  Here that is done for two
// broadcasting binary ops in a row, e.g. the affine tail (x * gamma) + beta
// of OpLayerNorm or the scaled, masked attention scores (scores + mask) / k
// of the GPT page's Attention section.  Per output element, with the local
// rules of each op (the chain rule, Autograd page, section 链式法则):
//   t      = a op1 b                 (recomputed, rounded as the forward did)
//   grad_t = d(t op2 c)/dt * g       g, g, g*c or g/c: one IEEE operation
//   grad_a = d(a op1 b)/da * grad_t  written densely (a has the output's shape)
//   grad_b += d(a op1 b)/db * grad_t summed over b's broadcast dims
//   grad_c += d(t op2 c)/dc * g      summed over c's broadcast dims
// grad_t and grad_a are the exact binary32 results the unfused ops would
// store; the two sums use the same Kahan-per-thread, fixed-tree scheme as
// k_reduce, and div's 1/b^2 (1/c^2) factor is applied once per output.
#pragma once

#include "zr_kernels.cuh"

namespace zr {

// Multiplier m with d(x op y)/dy * u = u * m (before div's post factor).
template <int OP>
__device__ __forceinline__ float dy_mult(float x) {
  if (OP == OP_ADD) return 1.0f;
  if (OP == OP_SUB) return -1.0f;
  return x;  // mul: u * x; div: u * x, then * -(1/y)^2 once per output
}

// One CTA = (kept index, row block, column block) of grad_b's plan, inner dim
// kept: thread (tx, ty) owns column vector tx of the block and adds rows ty,
// ty + ty_n, ... .  CSCALAR: c has one element and grad_c's per-CTA partial
// is a whole-CTA tree; otherwise grad_c shares grad_b's tiling.
template <int OP1, int OP2, bool CSCALAR>
__global__ void __launch_bounds__(kThreads, kOccChain)
k_chain_bwd(const __grid_constant__ ChainPlan cp) {
  constexpr int VEC = 4;
  constexpr bool kNeedT = OP2 == OP_MUL || OP2 == OP_DIV;
  const RedPlan& p = cp.r;
  pdl_trigger();
  extern __shared__ int64_t s_dyn[];
  const uint32_t table_rows = p.rows_per_blk < kMaxTileRows ? p.rows_per_blk : kMaxTileRows;
  int64_t* s_off = s_dyn;  // [table_rows][kMaxOperands]
  float* s_red = reinterpret_cast<float*>(s_dyn + kMaxOperands * table_rows);  // [kThreads * VEC]

  const RedCta cta = red_cta(p, blockIdx.x);
  int64_t base[kMaxOperands];
  decomp_offsets(p.kept, cta.kidx, base);
  const uint32_t row0 = cta.rblk * p.rows_per_blk;
  const uint32_t rleft = p.n_red - row0;
  const uint32_t nrows = rleft < p.rows_per_blk ? rleft : p.rows_per_blk;
  const uint32_t tx = threadIdx.x % p.tx;
  const uint32_t ty = threadIdx.x / p.tx;
  const uint32_t vcol_begin = cta.cblk * p.vcols_per_blk;
  const uint32_t vcol_end_raw = vcol_begin + p.vcols_per_blk;
  const uint32_t vcol_end = vcol_end_raw < p.nvcol ? vcol_end_raw : p.nvcol;
  const uint32_t ncs = vcol_end > vcol_begin + tx ? (vcol_end - vcol_begin - tx + p.tx - 1) / p.tx : 0;
  const uint32_t col = (vcol_begin + tx) * VEC;

  Kahan ab[VEC], ac[VEC], acs;
#pragma unroll
  for (int i = 0; i < VEC; ++i) { ab[i].init(); ac[i].init(); }
  acs.init();
  // b (and c when it has b's shape) is constant along the reduced rows: one
  // load per thread.
  Vec<VEC> bown, cown;
#pragma unroll
  for (int i = 0; i < VEC; ++i) { bown.v[i] = 0.f; cown.v[i] = 0.f; }
  float c0 = 0.f;

  for (uint32_t ch0 = 0; ch0 < nrows; ch0 += kMaxTileRows) {
    const uint32_t cleft = nrows - ch0;
    const uint32_t nch = cleft < kMaxTileRows ? cleft : kMaxTileRows;
    if (ch0 > 0) __syncthreads();
    for (uint32_t i = threadIdx.x; i < nch; i += blockDim.x) {
      int64_t off[kMaxOperands];
      decomp_offsets(p.red, row0 + ch0 + i, off);
#pragma unroll
      for (int k = 0; k < kMaxOperands; ++k) s_off[i * kMaxOperands + k] = off[k] + base[k];
    }
    __syncthreads();
    if (ch0 == 0) {
      pdl_wait();
      if (CSCALAR) c0 = __ldg(cp.c);
      if (ncs > 0) {
        bown = load_cols<VEC>(p.b, base[2], p.inner_stride[2], col, false);
        if (!CSCALAR) cown = load_cols<VEC>(cp.c, base[2], p.inner_stride[2], col, false);
      }
    }
    const uint32_t nrs = nch > ty ? (nch - ty + p.ty - 1) / p.ty : 0;
    const uint32_t items = ncs * nrs;  // ncs is 0 or 1 (one column vector per thread)
    constexpr int U = 4;
    for (uint32_t m0 = 0; m0 < items; m0 += U) {
      Vec<VEC> gv[U], av[U];
      uint32_t ri[U];
      bool ok[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        ok[u] = m0 + u < items;
        ri[u] = ty + (m0 + u) * p.ty;
        if (ok[u]) {
          const int64_t* ro = s_off + ri[u] * kMaxOperands;
          gv[u] = load_cols<VEC>(p.g, ro[0], p.inner_stride[0], col, p.stream_mask & 1);
          av[u] = load_cols<VEC>(p.a, ro[1], p.inner_stride[1], col, p.stream_mask & 2);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (!ok[u]) continue;
        Vec<VEC> dv;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          const float gg = gv[u].v[i], aa = av[u].v[i], bb = bown.v[i];
          const float cc = CSCALAR ? c0 : cown.v[i];
          const float gt = term_a<OP2>(gg, 0.f, cc);
          dv.v[i] = term_a<OP1>(gt, aa, bb);
          ab[i].add_prod(gt, dy_mult<OP1>(aa));
          const float tt = kNeedT ? fwd_op<OP1>(aa, bb) : 0.f;
          if (CSCALAR) acs.add_prod(gg, dy_mult<OP2>(tt));
          else ac[i].add_prod(gg, dy_mult<OP2>(tt));
        }
        store_cols<VEC>(p.d_out, s_off[ri[u] * kMaxOperands + kSlotOut], 1, col, dv);
      }
    }
  }

  // grad_b (and grad_c with b's shape): fixed tree over the ty row lanes of
  // each column vector, then one value per column to the output or to its
  // slot row [grad_b's nout | grad_c's nout] (CSCALAR: grad_b's nout only).
  const uint32_t lanes = p.tx * VEC;
  const uint32_t vc = vcol_begin + tx;
  const uint64_t j = uint64_t(cta.kidx) * p.ncol + uint64_t(vc) * VEC;
  for (int which = 0; which < (CSCALAR ? 1 : 2); ++which) {
    __syncthreads();
#pragma unroll
    for (int i = 0; i < VEC; ++i) s_red[ty * lanes + tx * VEC + i] = which == 0 ? ab[i].s : ac[i].s;
    for (uint32_t h = p.ty >> 1; h > 0; h >>= 1) {
      __syncthreads();
      if (ty < h) {
#pragma unroll
        for (int i = 0; i < VEC; ++i)
          s_red[ty * lanes + tx * VEC + i] =
              __fadd_rn(s_red[ty * lanes + tx * VEC + i], s_red[(ty + h) * lanes + tx * VEC + i]);
      }
    }
    __syncthreads();
    if (ty == 0 && vc < vcol_end) {
      Vec<VEC> r, f;  // sums, and div's -1/b^2 (-1/c^2) factors (1 otherwise)
      const bool div = which == 0 ? OP1 == OP_DIV : OP2 == OP_DIV;
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        r.v[i] = s_red[tx * VEC + i];
        f.v[i] = 1.0f;
        if (div) {
          const float rc = __frcp_rn(which == 0 ? bown.v[i] : cown.v[i]);
          f.v[i] = -__fmul_rn(rc, rc);
        }
      }
      if (p.nslots == 1) {
        if (div) {
#pragma unroll
          for (int i = 0; i < VEC; ++i) r.v[i] = __fmul_rn(r.v[i], f.v[i]);
        }
        store_cols<VEC>((which == 0 ? p.x_final : cp.c_final) + j, 0, 1, 0, r);
      } else {
        // Unscaled partials in slot row [grad_b | grad_c]; with a division
        // in the chain the rblk-0 CTAs also store every output's factor in a
        // row after the slots, and the second pass multiplies each total by
        // it (so no partial can overflow on its own).
        const uint64_t width = CSCALAR ? p.nout : 2 * p.nout;
        const uint64_t col0 = (which == 0 ? 0 : p.nout) + j;
        store_cols<VEC>(p.partial + uint64_t(cta.rblk) * width + col0, 0, 1, 0, r);
        if ((OP1 == OP_DIV || (!CSCALAR && OP2 == OP_DIV)) && cta.rblk == 0)
          store_cols<VEC>(p.partial + uint64_t(p.nslots) * width + col0, 0, 1, 0, f);
      }
    }
  }
  if (CSCALAR) {
    // grad_c = the total sum: one partial per CTA (whole-CTA fixed tree).
    __syncthreads();
    s_red[threadIdx.x] = acs.s;
    for (uint32_t h = blockDim.x >> 1; h > 0; h >>= 1) {
      __syncthreads();
      if (threadIdx.x < h) s_red[threadIdx.x] = __fadd_rn(s_red[threadIdx.x], s_red[threadIdx.x + h]);
    }
    if (threadIdx.x == 0) {
      float r = s_red[0];
      float f = 1.0f;
      if (OP2 == OP_DIV) {
        const float rc = __frcp_rn(c0);
        f = -__fmul_rn(rc, rc);
      }
      if (p.n_cta == 1) {
        *cp.c_final = OP2 == OP_DIV ? __fmul_rn(r, f) : r;
      } else {
        // Unscaled per-CTA partial; CTA 0 stores the factor after them.
        cp.c_partial[blockIdx.x] = r;
        if (OP2 == OP_DIV && blockIdx.x == 0) cp.c_partial[p.n_cta] = f;
      }
    }
  }
}

}  // namespace zr
