/*
 * zr_testing.h — host-only introspection hooks of the zr library, for tests
 * of the planner on machines without a GPU.  None of these touch device
 * memory or launch anything; data pointers are only inspected for alignment.
 * Return values are zr_status codes.
 */
#ifndef ZR_TESTING_H_
#define ZR_TESTING_H_

#include "zr.h"

#ifdef __cplusplus
extern "C" {
#endif

/* q = floor(n / d) through the kernels' multiply-high division (d >= 1). */
int zr_test_fastdiv(uint32_t d, uint32_t n, uint32_t* q);

/* JSON description of the plan zr_binary_fwd / zr_binary_bwd /
 * zr_sum_to_shape would launch for these arguments (NUL-terminated, up to
 * len bytes). */
int zr_test_describe_fwd(zr_op op, zr_tensor a, zr_tensor b, const float* out,
                         const int64_t* out_strides, char* buf, size_t len);
int zr_test_describe_bwd(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                         const float* grad_a, const float* grad_b, char* buf, size_t len);
/* The same for zr_binary_bwd_t with element type `dtype` (ZR_ERR_DTYPE for
 * an unknown one). */
int zr_test_describe_bwd_t(zr_dtype dtype, zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                           const void* grad_a, const void* grad_b, char* buf, size_t len);
int zr_test_describe_sum(zr_tensor in, int32_t ndim_out, const int64_t* sizes_out,
                         const float* out, char* buf, size_t len);

/* The same for zr_unary_fwd_t (x == NULL: in0 is x) and zr_unary_bwd_t
 * (in0 is grad_out, x is x) on `dtype` storage: "kernel" is "gelu_table" for
 * bfloat16 GeLU read from its table (k_gelu_bf16), else "flat" or
 * "elementwise".  `out` is the output (grad_x) with strides out_strides
 * (NULL: contiguous). */
int zr_test_describe_unary_t(zr_dtype dtype, zr_unary op, zr_tensor in0, const zr_tensor* x,
                             const void* out, const int64_t* out_strides, char* buf, size_t len);

/* JSON description of the route zr_chain_bwd would take ("fused" with its
 * plan, or "composed"), with its workspace sizes. */
int zr_test_describe_chain_bwd(zr_op op1, zr_op op2, zr_tensor grad_out, zr_tensor a,
                               zr_tensor b, zr_tensor c, const float* grad_a,
                               const float* grad_b, const float* grad_c, char* buf, size_t len);
/* Plan a chain backward and run its launch-time operand checks without
 * launching (as the zr_test_dry_run_* functions below). */
int zr_test_dry_run_chain_bwd(zr_op op1, zr_op op2, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                              zr_tensor c, const float* grad_a, const float* grad_b,
                              const float* grad_c);

/* Plan a call and run the launch-time operand checks without launching:
 * ZR_OK, an argument error, or ZR_ERR_CUDA if a kernel would read an operand
 * the plan does not provide. */
int zr_test_dry_run_fwd(zr_op op, zr_tensor a, zr_tensor b, const float* out,
                        const int64_t* out_strides);
int zr_test_dry_run_bwd(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                        const float* grad_a, const float* grad_b);
int zr_test_dry_run_sum(zr_tensor in, int32_t ndim_out, const int64_t* sizes_out,
                        const float* out);

/* Resident CTAs per SM of kernel `which` (0..27: elementwise forward add,
 * forward div, backward div, copy; reduction add inner-kept, sub
 * inner-reduced, mul inner-kept, div inner-reduced, sum-to-shape; split
 * forward; transpose; then the five reductions again in their cluster
 * variant; chain forward, fused chain backward with c shaped like b, the
 * same with c one element, chain forward with c one element; GeLU forward,
 * GeLU backward; flat forward add, flat GeLU forward, flat bfloat16 GeLU
 * forward; reduction add inner-kept with a three-batch staging ring in
 * shared memory; bfloat16 GeLU forward and backward by table) as the planner sizes grids for (*planned) and as the
 * CUDA runtime reports for the current device (*actual).  Needs a device:
 * ZR_ERR_CUDA without one; ZR_ERR_SIZE for an unknown `which`. */
int zr_test_occupancy(int which, int* planned, int* actual);

/* Walk every (CTA, thread item) of the planned forward kernel on the host and
 * record, per element visited, {out_offset, a_offset, b_offset} (element
 * units).  rec holds cap records of 3 int64; *nrec receives the count. */
int zr_test_emulate_fwd(zr_tensor a, zr_tensor b, const float* out, const int64_t* out_strides,
                        int64_t cap, int64_t* rec, int64_t* nrec);

/* Same for the backward plans: per element visited, 7 int64
 * {plan, g_offset, a_offset, b_offset, x_index, slot, d_offset}: plan is the
 * launch index; x_index the reduced gradient's element (-1 if none); slot its
 * partial slot; d_offset the densely written gradient's element (-1 if
 * none).  Offsets of operands the plan does not read are -1. */
int zr_test_emulate_bwd(zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                        const float* grad_a, const float* grad_b, int64_t cap, int64_t* rec,
                        int64_t* nrec);
/* The two walks above for plans on `dtype` storage (ZR_ERR_DTYPE for an
 * unknown type); offsets stay in elements. */
int zr_test_emulate_fwd_t(zr_dtype dtype, zr_tensor a, zr_tensor b, const void* out,
                          const int64_t* out_strides, int64_t cap, int64_t* rec, int64_t* nrec);
int zr_test_emulate_bwd_t(zr_dtype dtype, zr_op op, zr_tensor grad_out, zr_tensor a, zr_tensor b,
                          const void* grad_a, const void* grad_b, int64_t cap, int64_t* rec,
                          int64_t* nrec);

/* The two divisions of bfloat16 operands against the IEEE binary32 divide,
 * over every ordered pair of bfloat16 bit patterns (2^32 pairs, one kernel
 * on `stream`): the exact one (binary32 quotient rounded to nearest even,
 * without the general divide's slow path) bit for bit, and the one for
 * results stored as bfloat16 after both are rounded to bfloat16.  Two NaNs
 * count as equal.  out: four device words the caller sets to
 * {0, UINT64_MAX, 0, UINT64_MAX}; the kernel adds the number of differing
 * pairs of the first division to out[0] and lowers out[1] to the smallest
 * (x_bits << 16 | y_bits) among them, and likewise out[2], out[3] for the
 * second.  Returns ZR_ERR_NULL / ZR_ERR_DEVICE for a bad pointer,
 * ZR_ERR_CUDA if the launch fails. */
int zr_test_div_short_check(unsigned long long* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ZR_TESTING_H_ */
