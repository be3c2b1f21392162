/*
 * moe.h - C ABI of the GB300 (sm_103a) MXFP8-activation x MXFP4-weight
 * top-16 routed mixture-of-experts decode layer.
 *
 * What one call computes (pages "vllm.models.kimi_k3.nvidia.specialized_decode.
 * cutedsl.moe.experts" [experts] and "...cutedsl.moe.experts_runtime"
 * [runtime]): every token row x[t, :] (BF16) is quantized to MXFP8 (e4m3
 * codes, one E8M0 scale per 32 elements); for each of the token's 16 routed
 * experts e = ids[t, s], FC1 multiplies it by e's MXFP4 gate+up rows with FP32
 * accumulation, the hidden row SiLU(gate) * up is requantized to MXFP8, FC2
 * multiplies it by e's MXFP4 down rows, and the result is written as one BF16
 * row out[t, s, :] in the caller's top-16 order ([runtime] module docstring,
 * PersistentExperts.run; [experts] ExpertsKernel.store_hidden, ExpertsKernel.fc2).
 *
 * Conventions for every entry point:
 *  - Return value: 0 (MOE_OK) or one of enum moe_status. No entry point
 *    aborts the process; errors found before a launch leave nothing queued.
 *  - Device pointers are raw CUDA device addresses of the current device;
 *    host pointers are ordinary (preferably pinned) host memory. Stream
 *    arguments are cudaStream_t values passed as void*; NULL is the legacy
 *    default stream.
 *  - Ownership: the caller owns x, ids and out (and the weight arrays passed
 *    to moe_prepare, which may be freed once it returns). The handle owns
 *    every other buffer (repacked weights, activation plan, unit table,
 *    workspace) until moe_destroy.
 *  - A handle is bound to the device that was current at moe_prepare and
 *    serves one stream at a time: calls that overlap on the GPU race on its
 *    workspace. Every call that launches, copies or synchronizes returns
 *    MOE_ERR_ARG (nothing queued; moe_last_error_detail names both devices)
 *    when another device is current.
 */
#ifndef MXFP4_WEIGHT_MXFP8_GB300_MOE_H
#define MXFP4_WEIGHT_MXFP8_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_TOPK 16      /* routed experts per token */
#define MOE_UNIT_ROWS 8  /* pair rows per unit: the MMA's N */
#define MOE_MAX_BATCH 256
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_HIDDEN 16384
#define MOE_MAX_INTER 512
#define MOE_NOALLOC_SCRATCH_BYTES (8 << 20) /* static scratch of moe_run_noalloc */

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,            /* null/misaligned pointer, size out of range */
  MOE_ERR_UNSUPPORTED = 2,    /* not an sm_103 (GB300) device, grid not co-resident */
  MOE_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_TIMEOUT = 4, /* a bounded device-side wait ran out */
  MOE_ERR_DEVICE_IDS = 5,     /* an id out of [0, E) or repeated within a token */
  MOE_ERR_STATE = 6           /* call order: e.g. moe_copy_units before any grouping */
};

typedef struct moe_ctx* moe_handle;

/* Geometry of a prepared handle (moe_info). */
typedef struct moe_info_t {
  int experts, hidden, inter;
  int hidden_floor_rule;      /* 1: hidden requant uses floor(log2 amax) - 8 */
  int grid;                   /* persistent experts CTAs (one per SM) */
  int ring_stages;            /* weight-ring depth */
  int smem_bytes;             /* dynamic shared memory of the experts kernel */
  int stages_per_expert;      /* 16 KB weight + 1 KB scale stages per expert */
  int unit_capacity;          /* unit-table rows reserved (MOE_MAX_BATCH) */
  int hidden_image_bytes;     /* per-unit hidden image in the workspace */
  size_t weight_bytes;        /* repacked weight stages held by the handle */
  size_t workspace_bytes;     /* plan + unit table + workspace */
} moe_info_t;

/*
 * moe_prepare - take a copy of one layer's expert weights.
 * Source: [runtime] PersistentExperts.__init__ (weights w13, s13, w2, s2;
 * tp = 8 exactly when w13 has 768 rows) and scratch (model-owned workspace).
 *
 *   w13 uint8 [E, 2I, H/2]  e2m1 pairs, element 2i in the low nibble of byte i;
 *                           rows 0..I-1 are the gate rows, I..2I-1 the up rows
 *   s13 uint8 [E, 2I, H/32] E8M0 scale of each 32 consecutive k
 *   w2  uint8 [E, H, I/2]   e2m1 pairs (down projection)
 *   s2  uint8 [E, H, I/32]  E8M0
 * Each may be device or host memory (detected). Sizes: 1 <= E <= 1024,
 * H % 256 == 0 and H <= 16384, I % 32 == 0 and 32 <= I <= 512.
 * The hidden requant uses the floor rule iff 2I == 768, else the ceil rule.
 * Synchronous: repacks the weights into library-owned device memory (one
 * contiguous 17,408-byte block per 128-K stage of two 128-row tiles, scales
 * pre-tiled for the tensor core), allocates the plan, unit table and
 * workspace for batches up to MOE_MAX_BATCH, builds the TMA descriptor and
 * checks that the persistent grid fits one CTA per SM.
 * Errors: MOE_ERR_ARG (null out/pointers, sizes), MOE_ERR_UNSUPPORTED (the
 * current device fails moe_device_supported: the library holds sm_103a code
 * only), MOE_ERR_CUDA.
 * On error *out is NULL and nothing is leaked.
 */
int moe_prepare(moe_handle* out, const void* w13, const void* s13, const void* w2, const void* s2,
                int experts, int hidden, int inter);

/*
 * moe_quantize - MXFP8 activation plan of x.
 * Source: [experts] mx_block, plan_chunk and ExpertsPlanKernel (one E8M0
 * scale per 32 BF16 values; codes e4m3 of x * 2^-E). The scale rule is the
 * smallest E with max|x| <= 448 * 2^E (E = -127 for an all-zero block), so
 * no code saturates; codes round to nearest even, keeping the sign.
 *   x_bf16  device, BF16 [batch, H] row-major, 16-byte aligned
 *   1 <= batch <= MOE_MAX_BATCH
 * Asynchronous on `stream`; writes the handle's plan (read back with
 * moe_copy_plan). Errors: MOE_ERR_ARG, MOE_ERR_CUDA (launch).
 */
int moe_quantize(moe_handle h, const void* x_bf16, int batch, void* stream);

/*
 * moe_group - unit table of the routing ids.
 * Source: [experts] ExpertsKernel.group and ExpertsGroupKernel: experts in
 * ascending order; expert e's pairs p = token * 16 + slot, in token order,
 * fill ceil(n_e / 8) units of 8 rows, the last padded with -1.
 *   topk_ids  device, int32 [batch, 16]; ids must lie in [0, E) and be
 *             distinct within a token: a violating pair is dropped (its
 *             output row is not written) and the call reports
 *             MOE_ERR_DEVICE_IDS through moe_sync_status.
 * Asynchronous; also clears the per-call workspace counters. Read back with
 * moe_copy_units. Errors: MOE_ERR_ARG, MOE_ERR_CUDA.
 */
int moe_group(moe_handle h, const int32_t* topk_ids, int batch, void* stream);

/*
 * moe_run - the whole layer: quantize + group + experts + output epilogue.
 * Source: [runtime] PersistentExperts.run; [experts] ExpertsKernel (FC1 and
 * FC2 block-scaled FP4 x FP8 tensor-core stages with FP32 accumulation,
 * store_hidden, fc2).
 *   x_bf16     device BF16 [batch, H], 16-byte aligned
 *   topk_ids   device int32 [batch, 16] (same rules as moe_group)
 *   out_bf16   device BF16 [batch, 16, H], 16-byte aligned; row t*16+s is
 *              expert ids[t, s]'s output for token t
 * Asynchronous on `stream`; device-side errors surface through
 * moe_sync_status. A call of one or two tokens is one launch of the
 * small-batch kernel, any other call a prep grid and the experts kernel.
 * Launches are chained with programmatic dependent launch: the small-batch
 * kernel lets the next launch on the stream start while its own CTAs still
 * run, and a call reads its x and ids as soon as it starts. So x and ids
 * must not be the out_bf16 of the moe_run call just before on the stream
 * (every other producer is safe: a kernel of the caller, or
 * moe_run_combined, whose last launch lets the next start only when it has
 * ended). A call on the persistent grid kernel that follows another
 * handle's call on the same stream starts early: its prep grid writes this
 * handle's tables without waiting for the previous launch, and its experts
 * kernel streams weights while the previous call still runs, holding its
 * output rows until that call has ended. Every launch of this library lets
 * the next one start only after its own wait for the launch before it; a
 * caller's kernel launched between two calls with programmatic stream
 * serialization must likewise wait (griddepcontrol.wait) before it ends.
 * Errors: MOE_ERR_ARG (nulls, misalignment, batch range), MOE_ERR_CUDA.
 */
int moe_run(moe_handle h, const void* x_bf16, const int32_t* topk_ids, void* out_bf16, int batch,
            void* stream);

/*
 * moe_run_combined - moe_run, then the routing-weighted combine of each
 * token's 16 rows into one.
 * Source: [experts] ExpertsKernel.finalize (its single-GPU part: the 16 BF16
 * rows of a token are summed with their routing weights as FP32
 * multiply-adds in slot order and stored once per token).
 *   out[t, n] = bf16_rne(sum over s = 0..15 of w[t, s] * row[t, s, n]),
 * row[t, s, :] being the BF16 row moe_run would write for pair (t, s); pairs
 * the grouping dropped (bad or repeated ids) are left out of the sum.
 *   topk_weights  device, float32 [batch, 16], 16-byte aligned
 *   out_bf16      device, BF16 [batch, H]
 * The per-pair rows go to a handle-owned buffer, not to the caller. Same
 * stream semantics and errors as moe_run (a third kernel runs after the
 * experts kernel).
 */
int moe_run_combined(moe_handle h, const void* x_bf16, const int32_t* topk_ids,
                     const float* topk_weights, void* out_bf16, int batch, void* stream);

/*
 * moe_experts - kernels 3 and 4 alone: the persistent experts kernel and its
 * output epilogue, on the plan and unit table that moe_quantize and
 * moe_group (called in that order, with the same batch, on the same stream)
 * left in the handle. moe_quantize + moe_group + moe_experts computes
 * exactly what moe_run does. Each moe_experts call needs a moe_group of its
 * own before it: the grouping clears the per-call counters and flags that
 * the experts kernel consumes. Source: [runtime] PersistentExperts.group /
 * run (a unit-table kernel launched ahead of the experts kernel).
 *   out_bf16  device BF16 [batch, 16, H], 16-byte aligned
 * Errors: MOE_ERR_ARG, MOE_ERR_STATE (no plan or unit table of this batch),
 * MOE_ERR_CUDA.
 */
int moe_experts(moe_handle h, void* out_bf16, int batch, void* stream);

/*
 * moe_run_noalloc - moe_run for callers that cannot allocate device memory
 * when they run the layer. The pages have no counterpart to this call.
 *
 * Some runtimes hand all device memory to their own pool at start-up, or
 * must not call cudaMalloc on the decode path. This call computes exactly
 * what moe_run computes, with the same kernels, but takes none of its
 * per-call scratch (activation plan, unit table, split-K counters and
 * partial sums, hidden-vector images) from the handle's workspace: all of it
 * comes from one module-scope device array of MOE_NOALLOC_SCRATCH_BYTES
 * that every GPU loading this library keeps until the process exits. It
 * calls no cudaMalloc, cudaFree or other allocating routine. The caller
 * still passes x, ids and out (layouts as for moe_run) and a handle from
 * moe_prepare, the one-time set-up call that does allocate.
 *   - The scratch a call needs grows with batch, the layer's shape and the
 *     grid; a call that would need more than MOE_NOALLOC_SCRATCH_BYTES is
 *     rejected with MOE_ERR_ARG before any launch (moe_last_error_detail
 *     says how much it needed). The TP8 shard (H 3584, I 384, 384 experts)
 *     fits for batches up to 16 on a 152-SM GB300.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress with that device current); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, and the counters that
 *     must start at zero are cleared inside each call: calls that overlap on
 *     the GPU (other streams, other handles) race and corrupt each other.
 *   - Of the handle it reads the weights and settings and writes only the
 *     status word that moe_sync_status reads.
 *   - The array's address is looked up once per device and kept for the
 *     life of the process: a cudaDeviceReset (or any other teardown of the
 *     device's primary context) after the first call is not supported.
 * Asynchronous on `stream`; device-side errors surface through
 * moe_sync_status on the same handle. Errors: as moe_run, and
 * MOE_ERR_UNSUPPORTED on a device ordinal of 64 or more.
 */
int moe_run_noalloc(moe_handle h, const void* x_bf16, const int32_t* topk_ids, void* out_bf16,
                    int batch, void* stream);

/*
 * moe_run_host - moe_run on host buffers, on `stream`; synchronizes the
 * stream and returns the call's device status (as moe_sync_status). Pinned,
 * 16-byte aligned buffers on a GPU with native atomics on host memory (a
 * coherent GPU-CPU link, as on Grace) are used in place: the prep grid reads
 * x and ids from them and the experts kernel writes out into them, with no
 * copies. The first such call on a set of buffers and a batch captures the
 * two launches into a CUDA graph owned by the handle. Later calls with the
 * same buffers, batch and settings replay it as one graph launch. A new
 * set, or a changed timeout or test hook, captures again. Otherwise x and
 * ids are copied to handle-owned device buffers and out is copied back.
 *   x_host BF16 [batch, H], ids_host int32 [batch, 16], out_host BF16
 *   [batch, 16, H]. Errors: as moe_run, plus device-side status.
 */
int moe_run_host(moe_handle h, const void* x_host, const int32_t* ids_host, void* out_host,
                 int batch, void* stream);

/*
 * moe_sync_status - synchronize `stream` and return (and clear) the status
 * word the kernels write: MOE_OK, MOE_ERR_DEVICE_TIMEOUT (a bounded wait on
 * another CTA's result ran out; the kernel still finished) or
 * MOE_ERR_DEVICE_IDS. MOE_ERR_CUDA if the synchronization itself fails.
 */
int moe_sync_status(moe_handle h, void* stream);

/*
 * Read-back hooks (synchronous, for stage-by-stage checks):
 *  moe_copy_plan   codes uint8 [batch, H], scales uint8 [batch, H/32] of the
 *                  last quantize/run (batch <= that call's batch);
 *  moe_copy_units  unit count, experts int32 [capacity], rows int16
 *                  [capacity, 8] of the last group/run (MOE_ERR_ARG if the
 *                  count exceeds capacity);
 *  moe_copy_hidden hidden codes uint8 [units, 8, I] and scales uint8
 *                  [units, 8, I/32] of the last run, row r of unit u being
 *                  the unit's r-th pair (rows past the unit's last pair are
 *                  padding and hold stale bytes).
 * All write host memory; MOE_ERR_STATE before the producing call.
 */
int moe_copy_plan(moe_handle h, uint8_t* codes, uint8_t* scales, int batch);
int moe_copy_units(moe_handle h, int32_t* count, int32_t* experts, int16_t* rows, int capacity);
int moe_copy_hidden(moe_handle h, uint8_t* codes, uint8_t* scales, int units);

/*
 * moe_set_timeout - bound, in nanoseconds, of every device-side wait on
 * another CTA's hidden vector or on an mbarrier (default 2 s). After it
 * runs out the kernel records MOE_ERR_DEVICE_TIMEOUT and finishes without
 * waiting further. 0 restores the default.
 * moe_debug_withhold - test hook: the unit with this index never publishes
 * its hidden vector, so its consumers' waits run out (-1 = off, the
 * default). Used to check the bounded waits without faulting the GPU.
 * moe_debug_withhold_image - test hook for the grid kernel: the hidden
 * loader never hands this unit's hidden image to the MMA issuers, so their
 * mbarrier wait runs out and the CTA gives up (-1 = off, the default).
 * Checks the abort path: the call records MOE_ERR_DEVICE_TIMEOUT, finishes,
 * and the next call is unaffected. MOE_ERR_ARG below -1.
 * moe_debug_paths - which experts kernel small calls run on:
 * 1 (the default) the small-batch kernel for calls of one or two tokens
 * (two CTAs per SM, one of each of two consecutive calls; the unit table
 * derived from the routing ids in the kernel, every FC2 CTA summing the FC1
 * segment sums of its units itself) where the layer's shape fits it;
 * 0 the persistent grid kernel; 2 the cluster variant for one or two tokens
 * (one thread-block cluster of up to 8 CTAs per unit, partial sums and
 * hidden chunks through distributed shared memory) where the shape fits it;
 * 3 the small-batch kernel for calls of up to 8 tokens where the shape fits
 * it (measured no faster than the grid kernel at 3 to 8 tokens, hence not
 * the default there). Other calls, and calls whose path does not fit, run
 * on the grid kernel. The kernels cut the FC1 K range into split-K pieces at
 * different stages, so their FP32 sums are grouped differently and may
 * differ in the last bits. MOE_ERR_ARG for other values.
 * moe_kernel_path - the kernel a call of `batch` tokens runs on under the
 * current setting: 0 grid, 1 small-batch (under path 1 or 3), 2 cluster
 * variant (calls through moe_experts, which has no routing ids, never take
 * the small-batch kernel).
 * -MOE_ERR_ARG for a null handle or a batch outside [1, MOE_MAX_BATCH].
 */
int moe_set_timeout(moe_handle h, uint64_t nanoseconds);
int moe_debug_withhold(moe_handle h, int unit);
int moe_debug_withhold_image(moe_handle h, int unit);
int moe_debug_paths(moe_handle h, int path);
int moe_kernel_path(moe_handle h, int batch);

/*
 * moe_debug_kernel_span - measurement hook: with enable = 1, every later
 * launch of the experts kernel (cluster variant or grid) on this handle has
 * each CTA store its start and end time (%globaltimer, nanoseconds) into a
 * handle-owned array, overwriting the previous launch's (plain stores, no
 * synchronization between CTAs). 0 turns it off. Synchronizes the device and
 * clears the array when turned on.
 * moe_read_kernel_span - synchronizes the device and returns, in *span_ns,
 * the last recorded launch's span: the latest CTA end minus the earliest CTA
 * start. The launch overlaps the preceding prep grid (programmatic launch),
 * so its span starts while that grid still runs. Clears the array.
 * MOE_ERR_STATE if no launch was recorded since the last read.
 * Source: [runtime] PersistentExperts (one persistent launch per call; the
 * pages time it as part of the decode step). MOE_ERR_ARG for a null handle
 * or output, or another value of enable.
 */
int moe_debug_kernel_span(moe_handle h, int enable);
int moe_read_kernel_span(moe_handle h, uint64_t* span_ns);

/*
 * moe_cluster_size - the CTAs per thread-block cluster that a call of
 * `batch` tokens on this layer runs on: on the cluster variant the largest
 * size up to 8 of which one cluster per possible unit (min(E, 16 batch)) is
 * resident at once; 0 when the call does not run on it (more than two
 * tokens, shapes whose split-K pieces do not fit the variant's receive
 * buffer, too few resident clusters, or any moe_debug_paths setting but 2). -MOE_ERR_ARG for a null handle or a
 * batch outside [1, MOE_MAX_BATCH].
 */
int moe_cluster_size(moe_handle h, int batch);

int moe_info(moe_handle h, moe_info_t* info);

/* Free every buffer of the handle (synchronizes its device). NULL is a no-op. */
void moe_destroy(moe_handle h);

/* Static description of a status code. */
const char* moe_error_string(int status);

/* Text of the last failure seen by this thread (for MOE_ERR_CUDA,
 * MOE_ERR_UNSUPPORTED and some MOE_ERR_ARG diagnostics); empty if none. */
const char* moe_last_error_detail(void);

/*
 * moe_device_supported - whether a device with these properties runs this
 * library: compute capability 10.3 (sm_103, GB300; the library carries
 * sm_103a code only, and sm_100 parts lack it) with at least the experts
 * kernel's dynamic shared memory per block (cudaDeviceProp::
 * sharedMemPerBlockOptin). MOE_OK or MOE_ERR_UNSUPPORTED; pure, no CUDA
 * call. moe_prepare applies it to the current device. Source: [runtime]
 * PersistentExperts (one co-resident CTA per SM with the kernel's shared
 * memory) and the pages' sm_100-family tcgen05 kernels, here built for sm_103a.
 */
int moe_device_supported(int cc_major, int cc_minor, size_t smem_per_block_optin);

/*
 * moe_small_batch_build - which build of the small-batch kernel a call of
 * `batch` tokens (1..8) would run on a layer of this shape with `grid` CTAs
 * (the device's SM count, at most 256): 1 the packed build (one or two
 * tokens; the tokens' MXFP8 images of successive K chunks start 256 bytes
 * apart, which leaves room for a 3-slot weight ring in half an SM), 2 the
 * wide build (up to eight tokens, full 8-row images, 2-slot ring), 0 neither
 * fits the layer (its shared-memory layout, the landing of an item's segment
 * sums, or the FC2 split), so the grid kernel serves the call. Which calls
 * take the small-batch kernel at all is moe_debug_paths' setting. Pure host
 * arithmetic, no CUDA call. -MOE_ERR_ARG for sizes moe_prepare would refuse
 * or a batch or grid out of range. Source: [experts] ExpertsKernel (the
 * small-batch decode's one-launch path; the pages' kernel takes up to eight
 * tokens' rows in one MMA).
 */
int moe_small_batch_build(int experts, int hidden, int inter, int batch, int grid);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_WEIGHT_MXFP8_GB300_MOE_H */
