/*
 * igc_debug.h -- tuning and test hooks of libigc.so (not part of the
 * operations' interface in igc.h).
 *
 * These let a test or a tuning run force one schedule choice of the calls
 * that follow, so that every tile width, stage depth and int8 tensor path can
 * be checked against the oracle; none of them changes a result beyond fp32
 * rounding order (integer results are identical).  Each setting is
 * thread-local: it applies only to calls made by the thread that set it, so
 * a test or tuning thread cannot change the schedule of another thread's
 * calls.  A new thread starts with every hook at its default (0).
 */
#ifndef IGC_DEBUG_H
#define IGC_DEBUG_H

#include "igc.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Tuning and test hook: the output tile width (columns of B per CTA pair) of
 * every GEMM / convolution launched after this call.  0 (the default) picks it
 * per problem; 128, 224 or 256 force it where the operation is built for it
 * (the integer paths have 128 and 256; a width an operation lacks is ignored
 * for it).  Results do not depend on the width beyond fp32 rounding order
 * (integer results are identical).  Returns the previous setting, or -1 (and
 * changes nothing) for any other value.  Thread-local: it applies to the calls
 * of the thread that set it and to no other thread's.
 */
int igc_set_tile_width(int bn);

/*
 * Tuning and test hook: the k depth of the shared-memory pipeline stages of
 * the fp16 / bf16 GEMMs and the fp16 convolution launched after this call.
 * 0 (the default) picks it per problem: 64-deep stages (twice as many, more
 * bytes in flight) for a GEMM whose schedule is at most two rounds of tiles
 * over the CTA pairs, whose tiles fill at least a quarter of them and whose
 * K >= 2048, else 128-deep (always 128 for a convolution); 64 or 128 force
 * it.  The integer paths always use 128.  Results do not depend on the depth
 * beyond fp32 rounding order.  Returns the previous setting, or -1 (and
 * changes nothing) for any other value.  Thread-local: it applies to the calls
 * of the thread that set it and to no other thread's.
 */
int igc_set_stage_depth(int k);

/*
 * Selects the tensor path of gemm_s8_zp and gemm_s8_zp_dequant (the
 * prepare / run split and the convolutions always take the pre-pass form)
 * for calls made after this one:
 *  IGC_INT8_PATH_TCGEN05 (default): exact integers on the tcgen05 fp16 pipe
 *    after a pre-pass kernel that writes the operands shifted to [-128, 127]
 *    as fp16, with their row / column sums, into the workspace
 *    (gemm_s8_zp_prepare, then gemm_s8_zp_run).
 *  IGC_INT8_PATH_MMA_SYNC (gemm_s8_zp only; gemm_s8_zp_dequant takes the
 *    default): warp-level mma.sync m16n8k32 on the raw uint8 / int8 operands
 *    into int32 registers, raw row / column sums in the workspace's sum slots,
 *    the same correction and requantisation ([P1] §2.3's IMMA form).  Far
 *    slower on sm_103a, whose warp-level integer MMA rate is a fraction of the
 *    tcgen05 fp16 rate.
 *  IGC_INT8_PATH_FUSED: the same tcgen05 arithmetic with the shift and fp16
 *    widening done inside the GEMM kernel (int8 tiles by TMA, converter warps
 *    writing the fp16 operand stages, row / column sums in the same pass): no
 *    pre-pass and no workspace traffic, but about 1.8x the default's time at
 *    8192^3 on GB300, since every output tile converts its own operand panels.
 *  IGC_INT8_PATH_CONVERT: the default's GEMM kernel with the pre-pass folded
 *    into it: the CTAs' spare warps convert each 128-row block of the operands,
 *    1024 k at a time, once, into the workspace (jobs in the order the schedule
 *    first needs the blocks) while the tensor cores work, and the copies of a
 *    block wait for its completion flag.  One launch and no separate pass, but
 *    about 1.04x the default's time at 8192^3 on GB300: the conversion traffic
 *    shares each SM's path to L2 with the GEMM's own copies, and the first
 *    round waits for its blocks.  Needs K a multiple of 16 and both operands
 *    16-byte aligned with row strides that are multiples of 16; other calls
 *    take the default.  Its CTAs wait for conversion jobs that other CTAs of
 *    the same launch do, so it needs all of them resident at once: kernels on
 *    other streams that hold SMs delay it until they finish, and two such
 *    calls running at once on different streams can each hold the SMs the
 *    other's waiting CTAs need, until their bounded waits give up
 *    (IGC_ERR_DEVICE_TIMEOUT).  Use it from one stream at a time.
 * Every path gives bit-identical results.  Returns the previous setting, or
 * -1 (and changes nothing) for any other value.  Thread-local: it applies to
 * the calls of the thread that set it and to no other thread's.
 */
#define IGC_INT8_PATH_TCGEN05 0
#define IGC_INT8_PATH_MMA_SYNC 1
#define IGC_INT8_PATH_FUSED 2
#define IGC_INT8_PATH_CONVERT 3
int igc_set_int8_path(int path);

/*
 * Diagnostic: launches one CTA that waits on an mbarrier nothing ever
 * completes, with the current wait limit, and returns.  The wait gives up
 * after the limit and records IGC_ERR_DEVICE_TIMEOUT for
 * igc_check_device_status(); the context stays usable.  Used to test the
 * failure path without faulting or hanging the GPU.
 */
int igc_debug_wait_timeout_probe(igc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* IGC_DEBUG_H */
