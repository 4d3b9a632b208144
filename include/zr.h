/*
 * zr.h — C ABI of a GB300 (sm_103a) library of broadcasting elementwise
 * binary operators on strided fp32 tensors: forward, fused backward and
 * deterministic sum-to-shape.
 *
 * Semantics follow the "Zero" book (ismantic.github.io/zero):
 *   - Tensor page, section 形状与步长 (shape and strides): a tensor is a base
 *     pointer plus per-dimension sizes and element strides; element
 *     (i0, i1, ...) lives at base + sum_d i_d * stride_d.  Default strides are
 *     row-major, built from the last dimension ([2,3,4] -> [12,4,1]).
 *   - Operator page, section 广播 (broadcasting): shapes are compared from the
 *     last dimension; each pair must be equal, or one side 1, or one side
 *     missing (treated as 1).  A size-1 input dimension always reads
 *     coordinate 0.  Repetition in the forward pass is summation in the
 *     backward pass: dL/dx_j = sum over all outputs i that read x_j.
 *   - Operator page, section 逐元素算子 (elementwise ops): add, sub, mul, div;
 *     mul backward is (g*b, g*a).  GPU page, section OpAdd: add backward
 *     passes g to both inputs.  sub and div backward are not written out on
 *     the pages; this library uses the calculus rules (g, -g) and
 *     (g/b, -g*a/b^2).
 *   - Operator page, section 逐元素算子: shape and broadcast checks belong to
 *     the operator layer, not the kernels — every check here runs on the host
 *     before anything is launched.
 *   - GPU page, section Kernel 派发 (kernel dispatch): all operands of one op
 *     are on one device; up to eight dimensions are passed by value to the
 *     kernels (no metadata copies).
 *   - GPU page, section 异步执行 (asynchronous execution): every call only
 *     enqueues work on the caller's stream; success means "enqueued".
 *
 * Numerics.  Forward results are one IEEE binary32 operation per element,
 * round-to-nearest-even, no contraction, subnormals kept: bit-identical to
 * the same scalar C expression.  Gradients that receive exactly one term and
 * are one operation (add/sub copy or negation, mul g*b and g*a, div g/b) are
 * bit-identical too.  Reduced gradients, and div's -g*a/b^2, are within
 * 1e-5 * sum|terms| of the exact value per element; reductions use a fixed,
 * shape-determined order (no atomics), so results are bitwise reproducible
 * run to run on the same GPU model.
 *
 * Memory.  The library never allocates, frees or retains caller memory and
 * keeps no state between calls.  All pointers given for data must be device
 * memory of the current device, managed memory, or pinned (page-locked)
 * host memory that the device addresses at the same pointer (unified
 * addressing); kernels then read and write that host memory directly over
 * the host link.  Any other pointer (pageable host memory, another device's
 * memory, a pinned buffer with a different device alias) is ZR_ERR_DEVICE.
 * The caller owns the memory and the stream.
 *
 * Tracing.  With the environment variable ZR_TRACE set (and not "0") when
 * the library is first used, every zr_binary_fwd, zr_binary_bwd,
 * zr_binary_bwd_noalloc, zr_sum_to_shape, zr_unary_fwd and zr_unary_bwd call
 * (and their _t forms) that passes planning writes one
 * line "zr_trace <entry point> <plan as JSON>" to stderr before its device
 * checks and launches: the kernels, vector width, tiling, grid and
 * workspace it chose.
 */
#ifndef ZR_H_
#define ZR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as CUDA's cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* zr_stream_t;

/* Maximum rank of any operand (DimsArg-style, passed by value). */
#define ZR_MAX_DIMS 8

typedef enum { ZR_ADD = 0, ZR_SUB = 1, ZR_MUL = 2, ZR_DIV = 3 } zr_op;

typedef enum {
  ZR_OK = 0,
  ZR_ERR_NULL = -1,      /* required pointer is NULL, or op code unknown      */
  ZR_ERR_RANK = -2,      /* ndim < 0 or ndim > 8                               */
  ZR_ERR_SHAPE = -3,     /* shapes not broadcastable / wrong grad_out shape    */
  ZR_ERR_SIZE = -4,      /* negative size or stride, or index range overflow   */
  ZR_ERR_LAYOUT = -5,    /* output overlaps itself, or partially overlaps an
                            input or another output                           */
  ZR_ERR_DEVICE = -6,    /* pointer not addressable by the current device      */
  ZR_ERR_WORKSPACE = -7, /* workspace smaller than required                    */
  ZR_ERR_CUDA = -8,      /* a CUDA call or kernel launch failed                */
  ZR_ERR_DTYPE = -9      /* unknown element type (the _t entry points)         */
} zr_status;

/*
 * A strided fp32 tensor view (Tensor page, 形状与步长).
 *   data    : address of element (0, ..., 0); may be NULL only when the
 *             tensor is empty or the call does not read it (see below).
 *   ndim    : 0..8; ndim == 0 is a scalar (one element).
 *   sizes   : ndim sizes, each >= 0 (may be NULL when ndim == 0).
 *   strides : ndim element strides, each >= 0 (0 = expanded/broadcast view),
 *             or NULL for row-major contiguous.
 * The arrays are read during the call only.
 */
typedef struct {
  const void* data;
  int32_t ndim;
  const int64_t* sizes;
  const int64_t* strides;
} zr_tensor;

/*
 * zr_broadcast_shape — the broadcast rule (Operator page, 广播).
 * Writes the broadcast shape of (sizes_a[ndim_a]) and (sizes_b[ndim_b]) to
 * sizes_out[0 .. *ndim_out-1]; *ndim_out = max(ndim_a, ndim_b).  A size-0
 * dimension pairs with 0 or 1 (NumPy reading; the pages are silent).
 * Host only, launches nothing.  Errors: ZR_ERR_NULL, ZR_ERR_RANK,
 * ZR_ERR_SIZE (negative size), ZR_ERR_SHAPE (incompatible).
 */
int zr_broadcast_shape(int32_t ndim_a, const int64_t* sizes_a,
                       int32_t ndim_b, const int64_t* sizes_b,
                       int32_t* ndim_out, int64_t sizes_out[ZR_MAX_DIMS]);

/*
 * zr_binary_fwd — out = a op b with broadcasting (Operator page, 逐元素算子
 * and 广播).
 *   a, b        : inputs, any non-negative strides.
 *   out         : device buffer of the broadcast shape.
 *   out_strides : element strides of out (rank = broadcast rank), or NULL
 *                 for row-major contiguous.  out must not overlap itself.
 *                 out may alias an input exactly (same base, same shape as
 *                 out, same strides: in place); any other overlap with an
 *                 input is ZR_ERR_LAYOUT.
 * Empty outputs launch nothing.  Errors: ZR_ERR_NULL, ZR_ERR_RANK,
 * ZR_ERR_SHAPE, ZR_ERR_SIZE, ZR_ERR_LAYOUT, ZR_ERR_DEVICE, ZR_ERR_CUDA.
 * All checks happen before any launch: an error never writes to out.
 */
int zr_binary_fwd(zr_op op, zr_tensor a, zr_tensor b, float* out,
                  const int64_t* out_strides, zr_stream_t stream);

/*
 * zr_binary_bwd — fused backward of out = a op b (Operator page, 逐元素算子
 * and 广播; GPU page, OpAdd): one pass over grad_out computes
 *   grad_a = sum_to_shape(dL/da local terms, shape of a)
 *   grad_b = sum_to_shape(dL/db local terms, shape of b)
 * with local terms add (g, g), sub (g, -g), mul (g*b, g*a),
 * div (g/b, -g*a/b^2).
 *   grad_out : tensor of the broadcast shape, any strides.
 *   a, b     : the forward inputs; their sizes are always required.  Their
 *              data is read only where a term needs it (mul: b for grad_a, a
 *              for grad_b; div: b for grad_a, a and b for grad_b) and may be
 *              NULL otherwise.
 *   grad_a, grad_b : outputs, dense row-major in a's / b's own shape; either
 *              may be NULL to skip it.  They are written, not accumulated.
 *              An output may alias grad_out exactly (same shape, grad_out
 *              row-major); other overlaps are ZR_ERR_LAYOUT.
 *   workspace, workspace_bytes : scratch device memory for the two-pass
 *              reduction.  With workspace == NULL the call only stores the
 *              required size in *workspace_bytes and launches nothing.
 *              Otherwise *workspace_bytes is the size provided; if the
 *              required size is 0 any non-NULL pointer may be passed (it is
 *              not touched).  Workspace must be 16-byte aligned.
 * A reduced gradient of an empty grad_out is filled with zeros.
 * Errors: as zr_binary_fwd, plus ZR_ERR_WORKSPACE.
 */
int zr_binary_bwd(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                  float* grad_a, float* grad_b,
                  void* workspace, size_t* workspace_bytes, zr_stream_t stream);

/*
 * Size of the scratch array behind zr_binary_bwd_noalloc, in bytes.  Every
 * device that loads this library holds one such array until the process
 * exits.
 */
#define ZR_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * zr_binary_bwd_noalloc — the same fused backward as zr_binary_bwd, for
 * callers that cannot hand the library a workspace.  The pages have no
 * counterpart: this is an interface convenience, not part of the method.
 *
 * Who needs it: code that must not, or cannot, request device memory while
 * it runs — for example a callback inside a host framework that owns every
 * device allocation through its own pool and gives a library only the
 * tensors themselves, or a latency-critical path where cudaMalloc could
 * synchronise the device or fail under memory pressure.  This entry point
 * calls no allocator of any kind (no cudaMalloc, cudaFree, or allocating
 * library routine): the reduction's partial sums go to a fixed array of
 * ZR_STATIC_SCRATCH_BYTES bytes compiled into the library.
 *
 * Arguments, layout and results are those of zr_binary_bwd, without the
 * workspace.  A problem whose partial sums need more than
 * ZR_STATIC_SCRATCH_BYTES is rejected with ZR_ERR_WORKSPACE before anything
 * is launched (use zr_binary_bwd with a workspace for it; its workspace query
 * reports the size).
 *
 * The array is shared by every call on a device and keeps whatever the last
 * call left in it; nothing in it needs to start at zero, since each call
 * writes every partial it later reads.  Two calls whose work overlaps on the
 * GPU (e.g. on two streams without ordering between them) race on the array
 * and may return wrong gradients: order them, for instance by issuing them on
 * one stream.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  The address is remembered with the
 * device's context: after the context is replaced (cudaDeviceReset, for
 * example) the next call looks it up again, so make that call before any
 * capture too.
 */
int zr_binary_bwd_noalloc(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                          float* grad_a, float* grad_b, zr_stream_t stream);

/*
 * zr_sum_to_shape — OpSumToSize (Operator page, 广播): out[j] = sum of every
 * element of `in` whose coordinate maps to j when sizes_out is broadcast to
 * in's shape.  sizes_out must broadcast with in's shape to exactly in's shape
 * (else ZR_ERR_SHAPE).  out is dense row-major of sizes_out and must not
 * overlap `in` unless it aliases it exactly with no reduction.
 * Workspace protocol as zr_binary_bwd.
 */
int zr_sum_to_shape(zr_tensor in, int32_t ndim_out, const int64_t* sizes_out,
                    float* out, void* workspace, size_t* workspace_bytes,
                    zr_stream_t stream);

/*
 * Where and how zr_binary_bwd_ex writes one gradient.
 *   data        NULL: the gradient is not computed.
 *   strides     element strides over the input's shape (any non-negative
 *               layout that does not overlap itself); NULL: dense row-major.
 *   accumulate  nonzero: add the new gradient to the values already there,
 *               one binary32 addition per element (AccumulateGrad, Autograd
 *               page, section 反向传播: a gradient slot that already holds a
 *               value is summed in place, so a tensor reached by several
 *               paths gets the sum of their gradients).
 */
typedef struct {
  float* data;
  const int64_t* strides;
  int32_t accumulate;
} zr_grad;

/*
 * zr_binary_bwd_ex — zr_binary_bwd with a layout and a write mode per
 * gradient (zr_grad).  Results, numerics and the workspace protocol are
 * those of zr_binary_bwd; with accumulate, each element becomes
 * old + (the value zr_binary_bwd would write), rounded once.  A dense,
 * written gradient is written by the backward's own kernels; a strided or
 * accumulated gradient is formed densely in the workspace and then copied
 * into its layout, or added to the values there, by one more elementwise
 * pass, so the workspace query includes numel floats for it.  Layout errors (ZR_ERR_LAYOUT): a gradient that overlaps
 * itself, the other gradient or any input.  When grad_out is empty, written
 * gradients become zero and accumulated ones keep their values.
 */
int zr_binary_bwd_ex(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b, zr_grad grad_a,
                     zr_grad grad_b, void* workspace, size_t* workspace_bytes,
                     zr_stream_t stream);

/*
 * zr_chain_fwd — out = (a op1 b) op2 c, all three operands broadcast to one
 * output shape (broadcast(broadcast(a, b), c)).  The fused form of two of the
 * operators above in sequence: Operator page, section 融合 (fusion) — one
 * kernel launch, and the intermediate t = a op1 b never goes through memory,
 * while the mathematics stays that of the two operators (e.g. OpLayerNorm's
 * affine tail (x * gamma) + beta, or the GPT page's Attention section's masked
 * scores, here (scores + mask) / k).  t is rounded to binary32 before op2, so
 * every element is bit-identical to zr_binary_fwd(op2, zr_binary_fwd(op1, a,
 * b), c).  Layout, in-place and error rules are those of zr_binary_fwd (c is a
 * third input).
 */
int zr_chain_fwd(zr_op op1, zr_op op2, zr_tensor a, zr_tensor b, zr_tensor c, float* out,
                 const int64_t* out_strides, zr_stream_t stream);

/*
 * zr_chain_bwd — gradients of out = (a op1 b) op2 c given grad_out, by the
 * chain rule (Autograd page, section 链式法则): op2's local rules give
 * grad_t and grad_c; op1's rules applied to grad_t give grad_a and grad_b;
 * each gradient is summed back to its input's shape (Operator page, 广播).
 *
 *   grad_out  dense or strided, of the output shape (else ZR_ERR_SHAPE).
 *   a, b, c   the forward inputs.  Values are read only where the requested
 *             gradients need them: t = a op1 b (so a and b) when grad_c is
 *             requested and op2 is mul or div; b for grad_a and a for grad_b
 *             when op1 is mul or div (div's grad_b also b); c when op2 is mul
 *             or div.  Others may have data == NULL (sizes still required).
 *   grad_a, grad_b, grad_c
 *             dense row-major in a's, b's, c's shapes, or NULL to skip.  They
 *             must not overlap one another or any input (ZR_ERR_LAYOUT).
 *   workspace, workspace_bytes
 *             the zr_binary_bwd protocol: workspace == NULL queries the size
 *             (launches nothing); otherwise at least that many bytes, 16-byte
 *             aligned, owned by the caller, used in stream order.  The query
 *             sizes the route (below) that its own arguments select; a call
 *             whose pointers select the other route and need more workspace
 *             returns ZR_ERR_WORKSPACE without launching anything.
 *
 * When a has the output's shape, b is reduced with its innermost dim kept,
 * and c either has b's shape (both dense row-major) or one element, and all
 * three gradients are requested, one pass over grad_out writes grad_a and
 * sums grad_b and grad_c (plus a second pass over partial sums when the
 * reduction is split).  Any other layout runs the composition: t (when
 * needed) and grad_t are formed in the workspace, then op2's and op1's
 * backward passes, so the query covers numel(t) floats for each.
 * Numerics: grad_t and a dense grad_a are the binary32 values the two
 * unfused calls would produce (bit-identical); summed gradients are within
 * 1e-5 * sum|terms| per element, terms taken from the binary32 grad_t.
 */
int zr_chain_bwd(zr_op op1, zr_op op2, zr_tensor grad_out, zr_tensor a, zr_tensor b, zr_tensor c,
                 float* grad_a, float* grad_b, float* grad_c, void* workspace,
                 size_t* workspace_bytes, zr_stream_t stream);

/*
 * Unary elementwise ops.  The GPU page, section 逐元素运算 (elementwise
 * ops), lists GeLU and gradient scaling among the ops whose every output
 * element comes from the input element at the same position.
 *   ZR_SCALE  out = alpha * x, one IEEE binary32 multiply (bit-identical);
 *             backward grad_x = alpha * grad_out (bit-identical).
 *   ZR_GELU   out = x * Phi(x), the exact GeLU (the pages give no formula;
 *             Phi is the standard normal CDF, computed as erfc(-x/sqrt 2)/2),
 *             alpha unused; backward grad_x = grad_out * (Phi(x) + x phi(x)),
 *             phi the standard normal density.  Within
 *             (16 + 2x^2) * 2^-24 * |exact| + 2^-120 per element forward, and
 *             (16 + 2x^2) * 2^-24 * |g| (Phi(x) + |x| phi(x)) + 2^-120
 *             backward (the derivative's two terms cancel near x = -0.75;
 *             the x^2 term is the binary32 argument of erfc, whose tail
 *             amplifies relative argument error by about x^2).
 */
typedef enum { ZR_SCALE = 0, ZR_GELU = 1 } zr_unary;

/*
 * zr_unary_fwd — out = op(x), out of x's shape with out_strides (NULL:
 * dense row-major).  Any input strides; out may alias x exactly (same
 * layout); other overlap is ZR_ERR_LAYOUT.  Errors and asynchrony as
 * zr_binary_fwd.
 */
int zr_unary_fwd(zr_unary op, float alpha, zr_tensor x, float* out, const int64_t* out_strides,
                 zr_stream_t stream);

/*
 * zr_unary_bwd — grad_x = grad_out * op'(x), written in grad_x_strides (NULL:
 * dense row-major) over x's shape (which must equal grad_out's, else
 * ZR_ERR_SHAPE).  ZR_SCALE reads no x values (x.data may be NULL).
 */
int zr_unary_bwd(zr_unary op, float alpha, zr_tensor grad_out, zr_tensor x, float* grad_x,
                 const int64_t* grad_x_strides, zr_stream_t stream);

/*
 * Element types of the _t entry points below.  ZR_F32 is binary32 (the
 * entry points above).  ZR_BF16 is bfloat16 storage: every operand and
 * output is bf16 (2 bytes, strides still in elements), arithmetic is the
 * binary32 arithmetic above, and each stored element is rounded once to bf16,
 * to nearest with ties to even.  Because binary32 carries at least
 * 2 * 8 + 2 significand bits, a forward element or a one-operation gradient
 * equals the exact result rounded to bf16, bit for bit; a summed gradient is
 * within 1e-5 * sum|terms| + 2^-7 * |its exact value| (one bf16 unit in the
 * last place: the binary32 sum and the exact one may round to neighbouring
 * bf16 values).
 * Partial sums in the workspace stay binary32, so the workspace protocol and
 * sizes are those of the float entry points.  Same-layout in-place outputs,
 * errors and asynchrony are as above; unknown dtype: ZR_ERR_DTYPE.
 */
typedef enum { ZR_F32 = 0, ZR_BF16 = 1 } zr_dtype;

/* zr_binary_fwd on `dtype` storage. */
int zr_binary_fwd_t(zr_dtype dtype, zr_op op, zr_tensor a, zr_tensor b, void* out,
                    const int64_t* out_strides, zr_stream_t stream);
/* zr_binary_bwd on `dtype` storage. */
int zr_binary_bwd_t(zr_dtype dtype, zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                    void* grad_a, void* grad_b, void* workspace, size_t* workspace_bytes,
                    zr_stream_t stream);
/* zr_sum_to_shape on `dtype` storage. */
int zr_sum_to_shape_t(zr_dtype dtype, zr_tensor in, int32_t ndim_out, const int64_t* sizes_out,
                      void* out, void* workspace, size_t* workspace_bytes, zr_stream_t stream);
/* zr_unary_fwd on `dtype` storage.  ZR_SCALE is bit-identical to the exact
 * product rounded to bf16.  ZR_GELU on bf16 evaluates erfc with a shorter
 * polynomial fitted for bf16 results (relative error below 2^-16.3); each
 * result is within half a bf16 unit in the last place of the exact value plus
 * 2^-14 of its size plus 2^-120 (backward: 2^-14 of
 * |g| (Phi(x) + |x| phi(x))), so it is the correctly rounded value except
 * next to a rounding boundary.  Large calls over a layout that flattens to at
 * most two dims (at least 32,768 elements per SM) read the results from a
 * table in shared memory that each thread block fills with the same
 * arithmetic, for the 8192 values 2^-24 <= |x| < 256, and evaluate the others
 * in place: the results do not depend on which path ran. */
int zr_unary_fwd_t(zr_dtype dtype, zr_unary op, float alpha, zr_tensor x, void* out,
                   const int64_t* out_strides, zr_stream_t stream);
/* zr_unary_bwd on `dtype` storage, with the same accuracy as zr_unary_fwd_t. */
int zr_unary_bwd_t(zr_dtype dtype, zr_unary op, float alpha, zr_tensor grad_out, zr_tensor x,
                   void* grad_x, const int64_t* grad_x_strides, zr_stream_t stream);

/* Static, human-readable name of a status code. */
const char* zr_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ZR_H_ */
