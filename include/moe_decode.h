/*
 * moe_decode.h -- C ABI of the GB300 small-batch MoE decode layer step.
 *
 * One call computes, for M = 1..16 token rows, the MoE block of a decoder layer:
 *
 *   1. router GEMV      l[m,e] = sum_h x[m,h] Wr[e,h]          (bf16 in, fp32 acc)
 *   2. top-k select     the k largest l[m,:], ties to the lower expert id, with
 *                       renormalised weights w_j = exp(l_j - l_max) / sum_sel exp(.)
 *                       (= softmax over all experts -> top-k -> renormalise); or
 *                       the bias-corrected sigmoid rule (see moe_score)
 *   3. routed experts   h = silu(Wg_e x) * (Wu_e x),  y_e = Wd_e h   (fp32)
 *   4. shared experts   the same SwiGLU MLP with the shared weights, weight 1
 *   5. combine          out = bf16_rne(r + routed_scale * sum_j w_j y_{e_j} + sum_s y_s)
 *
 * Sources: the Ling-3.0-flash batch-1 decode blog (LMSYS) -- section "PDL:
 * stacking the latency floors of small kernels" (router chain norm -> gate
 * matvec -> top-k; the MoE chain up-GEMM -> activation -> down-GEMM -> combine;
 * the combine is one fp32 sum times a scale with a single final cast), section
 * "Two fusions and a retune" (silu(gate) * up in fp32 inside the up-GEMM, w13 =
 * [gate; up]), section "bf16 router gate and lm_head" (bf16 router matvec), and
 * its model table (512 routed + 1 shared expert, top-8(+1), moe_intermediate 768,
 * hidden 2560); "Muse Spark Open Ultrafast", section "The model" (8 of 256
 * experts, NVFP4 expert weights); "SGLang Low-Latency Mode: kernels and
 * runtime", section "Low-Latency-Specific Optimizations" item 3 (at most eight
 * rows: expert row sets placed by bitmap and population count). The pages do not
 * fix the scoring rule; softmax -> top-k -> renormalise is the default, and a
 * bias-corrected sigmoid rule is the second (moe_score).
 *
 * Threading: a handle may be used from one host thread at a time. Runs on one
 * handle must not overlap on the GPU (they share the handle's scratch); issue
 * them on one stream, or order the streams.
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_DECODE_ABI_VERSION 3

/* A cudaStream_t. NULL means the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, M out of range, bad option */
  MOE_ERR_UNSUPPORTED = 2,    /* a config outside the supported shapes (see below)   */
  MOE_ERR_CUDA = 3,           /* a CUDA runtime call failed                          */
  MOE_ERR_DEVICE_TIMEOUT = 4, /* a device-side wait ran past its limit (see get_status) */
  MOE_ERR_OOM = 5             /* device allocation failed in create                  */
} moe_status;

typedef enum moe_wdtype {
  MOE_W_BF16 = 0,      /* expert weights bf16                                     */
  MOE_W_NVFP4 = 1,     /* expert weights e2m1 codes + e4m3 block-16 scales + fp32 */
  MOE_W_FP8_BLOCK = 2  /* expert weights e4m3 + one fp32 scale per 128 x 128 block
                          (Ling-3.0-flash blog, "Where the time goes now": fp8
                          weights halve the bytes; block 128)                     */
} moe_wdtype;

/*
 * Router scoring rules. The pages do not fix one: the Ling blog's router top-k
 * "prefetches its bias" (section "PDL: stacking the latency floors of small
 * kernels"), which points at a bias-corrected router; softmax -> top-k ->
 * renormalise is the default reading.
 */
typedef enum moe_score {
  MOE_SCORE_SOFTMAX_TOPK_RENORM = 0, /* softmax over E -> top-k -> renormalise:
                                        w_j = exp(l_j - l_max) / sum_sel exp(l_i - l_max) */
  MOE_SCORE_SIGMOID_BIAS = 1         /* s_e = sigmoid(l_e); the k largest s_e + bias_e are
                                        selected (ties to the lower id); w_j = s_j / sum_sel s_i.
                                        The bias steers the choice only.                   */
} moe_score;

/*
 * Layout of the down matrices (w2, sh_w2 and, for FP8, their block scales).
 * MOE_W2_I_H stores each expert's down matrix transposed, so that the down
 * weights of one intermediate row are one contiguous row. A handle built with it
 * runs the split-K single kernel: each CTA applies the down projection to the
 * intermediate rows it computed itself and the output is a fixed-order sum of
 * every CTA's partial sums ("Muse Spark Open Ultrafast", section "A new tensor
 * parallelism": the second expert GEMM split on the intermediate dimension with
 * one reduction at the end, here across the CTAs of one GPU). The layer computed
 * is the same; the order of the down projection's sums differs.
 */
typedef enum moe_w2_layout {
  MOE_W2_H_I = 0,  /* w2 [E, H, I] (output rows), the default                      */
  MOE_W2_I_H = 1   /* w2 [E, I, H] (intermediate rows); bf16 or FP8, hidden <= 3072,
                      MOE_SCHED_PERSISTENT only                                     */
} moe_w2_layout;

typedef enum moe_sched {
  MOE_SCHED_PERSISTENT = 0, /* one cooperative kernel; phases hand off through tagged data */
  MOE_SCHED_PDL_CHAIN = 1,  /* three kernels (router, gate/up, down) chained with PDL      */
  MOE_SCHED_CHAIN = 2       /* the same three kernels without PDL (plain stream order)     */
} moe_sched;

/*
 * Layer configuration. Supported (create/config_check return MOE_ERR_UNSUPPORTED
 * otherwise):
 *   2 <= num_experts <= 1024, even;  1 <= top_k <= min(16, num_experts);
 *   0 <= num_shared <= 4;  1 <= max_rows <= 16 (a run of more than 8 rows launches
 *   row groups of at most 8, one after another: the wider verify batch of the Muse
 *   Spark page, "Speculative decoding", checks 16 tokens per step);
 *   bf16:  hidden % 8 == 0, 64 <= hidden <= 4096; inter % 8 == 0 and inter / 8
 *          either a power of two <= 32 or a multiple of 32 no larger than 384;
 *   nvfp4: hidden % 256 == 0, 256 <= hidden <= 4096; inter % 256 == 0, inter <= 12288;
 *   fp8:   hidden % 128 == 0, hidden <= 4096; inter % 128 == 0 and inter / 8 as for bf16;
 *   routed_scale finite; rms_eps > 0 when pre_rmsnorm.
 */
typedef struct moe_decode_config {
  int32_t hidden;      /* H: model width                                      */
  int32_t inter;       /* I: expert intermediate size (shared experts too)    */
  int32_t num_experts; /* E: routed experts                                   */
  int32_t top_k;       /* k: experts per row                                  */
  int32_t num_shared;  /* S: always-on shared experts (weight 1)              */
  int32_t max_rows;    /* largest M passed to run                             */
  int32_t wdtype;      /* moe_wdtype                                          */
  int32_t score;       /* moe_score                                           */
  float routed_scale;  /* multiplies the routed sum (1.0 when unused)         */
  int32_t pre_rmsnorm; /* 1: the layer input is bf16(RMSNorm(x)), gamma = 1  */
  float rms_eps;       /* RMSNorm epsilon (1e-6)                              */
  int32_t sched;       /* moe_sched                                           */
  int32_t w2_layout;   /* moe_w2_layout                                       */
} moe_decode_config;

/*
 * Weight pointers: device memory, BORROWED (the caller keeps ownership and must
 * keep them alive and unchanged until destroy). Every pointer 16-byte aligned.
 * Row-major, no padding:
 *   router_w        bf16  [E, H]
 *   bf16:   w13     bf16  [E, 2I, H]   rows 0..I-1 gate, I..2I-1 up
 *           w2      bf16  [E, H, I]
 *   nvfp4:  w13     uint8 [E, 2I, H/2] e2m1 codes, element 2i in the low nibble
 *           w13_scale uint8 [E, 2I, H/16] e4m3 scale per 16 consecutive elements
 *           w13_gscale fp32 [E, 2]     tensor scale of the gate rows, of the up rows
 *           w2      uint8 [E, H, I/2], w2_scale uint8 [E, H, I/16], w2_gscale fp32 [E]
 *   fp8:    w13     uint8 [E, 2I, H]   e4m3 codes; w13_scale fp32 [E, 2I/128, H/128]
 *           w2      uint8 [E, H, I]    e4m3 codes; w2_scale  fp32 [E, H/128, I/128]
 *           (w = e4m3(code) * scale[row / 128][col / 128]; gscale pointers unused)
 *   w2_layout MOE_W2_I_H: w2 bf16 [E, I, H]; fp8 w2 uint8 [E, I, H] with
 *           w2_scale fp32 [E, I/128, H/128] (the transpose of the tensors above)
 *   sh_*            the same for the S shared experts (leading dim S)
 *   router_bias     fp32  [E] selection bias, 4-byte aligned (MOE_SCORE_SIGMOID_BIAS)
 * Unused pointers (scales for bf16, shared for S = 0, the bias under softmax
 * scoring) may be NULL.
 */
typedef struct moe_decode_weights {
  const void* router_w;
  const void* w13;
  const void* w2;
  const void* w13_scale;
  const void* w2_scale;
  const float* w13_gscale;
  const float* w2_gscale;
  const void* sh_w13;
  const void* sh_w2;
  const void* sh_w13_scale;
  const void* sh_w2_scale;
  const float* sh_w13_gscale;
  const float* sh_w2_gscale;
  const float* router_bias;
} moe_decode_weights;

typedef struct moe_decode_handle moe_decode_handle;

/*
 * Validates a config on the host. Makes no CUDA call. This is the "guard" of the
 * SGLang Low-Latency Mode page, section "Plugin System: Design and Integration":
 * declared requirements are checked before any weight is touched, so an
 * unsupported configuration fails early. The shapes it accepts cover the pages'
 * layers: Ling-3.0-flash (model table: hidden 2560, 512 routed + 1 shared expert,
 * top-8, moe_intermediate 768) and Muse Spark ("The model": 8 of 256 experts, NVFP4).
 */
moe_status moe_decode_config_check(const moe_decode_config* cfg);

/*
 * The launch layout create would plan for cfg on a device with `sms` SMs and
 * `smem_optin` bytes of opt-in shared memory per block, computed on the host
 * (no CUDA call). `interleaved` = 1 asks for the slot-interleaved single kernel's
 * layout, 2 for the expert-range kernel's (MOE_ERR_UNSUPPORTED when it does not
 * fit), 0 for the phase-ordered kernels'. A config with w2_layout MOE_W2_I_H has
 * one layout, the split-K kernel's (interleaved must be 0). All fields in bytes
 * or counts; filled only on MOE_OK.
 */
typedef struct moe_decode_plan_info {
  int32_t smem_bytes;        /* dynamic shared memory per CTA (incl. alignment slack)   */
  int32_t ring_slots;        /* weight ring slots                                         */
  int32_t slot_bytes;        /* bytes per slot                                            */
  int32_t extra_slots;       /* gate/up ring slots carved from the idle h area             */
  int32_t down_slot_in_x;    /* 1: one more down-phase slot in the x area                  */
  int32_t pairs_per_stage;   /* gate/up row pairs per stage                                */
  int32_t router_pairs_per_stage;
  int32_t down_rows_per_stage;
  int32_t h_pairs;           /* (expert, row) h rows staged in shared memory at once       */
  int32_t h_buffers;         /* 1 or 2 h batch buffers                                    */
  int32_t h_per_slot;        /* 1: per-slot h fetches (phase-ordered, NVFP4)               */
  int32_t slots_max;         /* union slots at most: shared + min(E, max_rows * k)         */
  int32_t pairs_max;         /* (expert, row) pairs at most                                */
  int32_t lag;               /* interleaved: down stage of slot s after the gate/up of s+lag */
  int32_t down_h_offset;     /* interleaved: h rows' offset in a down stage's slot        */
  int32_t threads;           /* threads per CTA                                           */
  int32_t h_rows_max;        /* split-K (w2_layout MOE_W2_I_H): h rows one CTA holds      */
  int32_t down_t_rows_per_stage; /* split-K: transposed down rows per stage             */
} moe_decode_plan_info;
moe_status moe_decode_plan(const moe_decode_config* cfg, int32_t sms, int32_t smem_optin, int32_t interleaved,
                           moe_decode_plan_info* out);

/*
 * Builds a handle for the current CUDA device -- the "build" step of the SGLang
 * Low-Latency Mode page, section "Plugin System: Design and Integration":
 * execution resources are set up once at initialisation and reused by every
 * request. It validates cfg and the weight
 * pointers, allocates the handle's device scratch (control words, tagged
 * logits and intermediate activations, host-call staging buffers) and plans the
 * launch shape from the device's SM count and shared memory. Copies nothing and
 * repacks no weight. On error *out is NULL and nothing stays allocated.
 * MOE_ERR_UNSUPPORTED also when cfg passes moe_decode_config_check but its layout
 * does not fit the device's shared memory (the largest H x I at max_rows 6..8;
 * moe_decode_plan tells in advance).
 */
moe_status moe_decode_create(const moe_decode_config* cfg, const moe_decode_weights* w,
                             moe_decode_handle** out);

/*
 * Enqueues one layer step on `stream`; returns without waiting. The step is the
 * router chain (norm -> gate matvec -> top-k) and the MoE chain (up-GEMM ->
 * activation -> down-GEMM -> combine) of the Ling-3.0-flash batch-1 decode blog,
 * section "PDL: stacking the latency floors of small kernels", fused into one
 * persistent kernel or chained with programmatic dependent launch (cfg.sched);
 * the "runtime" step of the plugin section above (a dispatch that a CUDA graph
 * can record once and replay).
 *   x        bf16 [M, H] device, layer input (normalised inside when pre_rmsnorm)
 *   residual bf16 [M, H] device
 *   out      bf16 [M, H] device; may be the same buffer as residual and/or x
 *   m_rows   1 <= M <= cfg.max_rows
 *   topk_idx int32 [M, k] device or NULL: chosen experts, descending weight
 *   topk_w   fp32  [M, k] device or NULL: their renormalised weights
 * All device pointers 16-byte aligned. Allocates nothing, never synchronises and
 * never reads device memory back, so it can be captured in a CUDA graph. Returns
 * only argument and launch errors; device-side wait timeouts are reported by
 * moe_decode_get_status.
 */
moe_status moe_decode_run(moe_decode_handle* h, const void* x, const void* residual, void* out,
                          int32_t m_rows, int32_t* topk_idx, float* topk_w, moe_stream_t stream);

/*
 * The same step from host memory: copies x and residual (bf16 [M, H], host; one
 * copy when they are the same buffer) into the handle's staging buffers, runs,
 * brings the device status words, topk_idx / topk_w and out back in one
 * device-to-host copy into a pinned staging block, synchronises `stream` and
 * copies out (and topk_idx / topk_w when not NULL, host) from there. Host buffers
 * should be pinned for speed; pageable memory works. Returns the device status as
 * get_status does.
 */
moe_status moe_decode_run_host(moe_decode_handle* h, const void* x_host, const void* residual_host,
                               void* out_host, int32_t m_rows, int32_t* topk_idx_host,
                               float* topk_w_host, moe_stream_t stream);

/*
 * Synchronises `stream`, reads and clears the handle's device status word. Every
 * device-side wait is bounded (the Muse Spark page, "Megakernel internals": a
 * missed deadline stops the launch instead of hanging the server), and a wait that
 * gives up is reported here.
 * MOE_ERR_DEVICE_TIMEOUT means some device-side wait of an earlier run on this
 * handle gave up after the wait limit; that run's outputs are undefined.
 */
moe_status moe_decode_get_status(moe_decode_handle* h, moe_stream_t stream);

/* Options for moe_decode_set_option / moe_decode_get_info. */
enum {
  MOE_OPT_SCHED = 1,           /* moe_sched of later runs                           */
  MOE_OPT_WAIT_TIMEOUT_NS = 2, /* device wait limit in ns (default 1e9)             */
  MOE_OPT_TEST_FLAGS = 3,      /* testing only: 1 = router results are never published,
                                  so every wait on them runs into the limit          */
  MOE_OPT_RING_SLOTS = 4,      /* shared-memory ring slots used, 2 .. the planned count */
  MOE_OPT_STAMPS = 5,          /* device pointer (as int64) to a uint64 buffer of
                                  MOE_INFO_GRID x 24 words, or 0: each CTA stores the
                                  %globaltimer ns at its phase boundaries (profiling)  */
  MOE_OPT_INTERLEAVE = 6,      /* MOE_SCHED_PERSISTENT runs with the slot-interleaved
                                  kernel (gate/up items and down stages alternate
                                  slot by slot) when its layout fits and: 1 (default)
                                  for bf16 weights and one token row, where it
                                  measured faster; 2 always (bf16 and FP8); 0 never (the phase-
                                  ordered kernel). get_info: the mode, 0 when the
                                  interleaved layout does not fit.                   */
  MOE_OPT_FLAT = 7,            /* MOE_SCHED_PERSISTENT runs with the expert-range
                                  kernel (each CTA owns a contiguous range of the
                                  routed experts' rows and output blocks; bf16
                                  weights, at most one shared expert) when its layout
                                  fits and: 0 (default) never; 1 for one token row;
                                  2 always. It measured slower than the other
                                  single kernels on GB300. It takes precedence over
                                  MOE_OPT_INTERLEAVE. get_info: the mode, 0 when the
                                  layout does not fit.                               */
  MOE_OPT_PREFETCH_EXPERTS = 8, /* 0 (default) .. 16: while a run routes, its producer
                                  warps pull into L2 the weights of this many experts
                                  that the handle's previous run used most (most token
                                  rows, ties to the lower id; with one row, the first
                                  selected), each CTA its 1/grid share ("Muse Spark Open
                                  Ultrafast", section "Speculative expert prefetching":
                                  consecutive steps tend to route alike). Results do
                                  not change. Phase-ordered, interleaved, chained and
                                  split-K kernels; the expert-range kernel ignores it. */
  MOE_INFO_GRID = 16,          /* CTAs per kernel                                   */
  MOE_INFO_THREADS = 17,       /* threads per CTA                                   */
  MOE_INFO_SMEM = 18,          /* dynamic shared memory per CTA, bytes              */
  MOE_INFO_RING_SLOTS = 19,    /* shared-memory weight ring: slots                  */
  MOE_INFO_SLOT_BYTES = 20,    /*                            bytes per slot         */
  MOE_INFO_KERNELS_PER_RUN = 21,
  MOE_INFO_SCRATCH_BYTES = 22,
  MOE_INFO_INTERLEAVED_ROWS = 23, /* bit m-1 set: a run of m rows under the current
                                    schedule and options takes the slot-interleaved
                                    kernel                                         */
  MOE_INFO_FLAT_ROWS = 24,       /* the same for the expert-range kernel            */
  MOE_INFO_SPLIT_K = 25,         /* 1: the handle runs the split-K kernel (w2_layout
                                    MOE_W2_I_H)                                       */
  MOE_INFO_PREDICTED = 32        /* + i (i < 16): the i-th expert the next run
                                    prefetches, -1 for none. Waits for the device
                                    (cudaDeviceSynchronize) and reads device memory.  */
};
moe_status moe_decode_set_option(moe_decode_handle* h, int32_t option, int64_t value);
moe_status moe_decode_get_info(moe_decode_handle* h, int32_t what, int64_t* value);

/*
 * moe_decode_run_static -- the same layer step without a handle, allocating
 * nothing. The pages have no counterpart; this is a convenience of the library.
 *
 * For callers that cannot allocate device memory: code hosted by a framework
 * that owns all device memory and forbids allocations after start-up, code on a
 * latency-critical thread that must not take cudaMalloc's implicit device
 * synchronisation or driver locks, or callers that cannot keep a handle alive
 * between calls. The caller still passes the weights, inputs and outputs
 * (device pointers, same meaning and layout as for moe_decode_create and
 * moe_decode_run; cfg->sched is ignored: the single-kernel schedule runs).
 *
 * Scratch: a file-scope device array of MOE_DECODE_STATIC_SCRATCH_BYTES that
 * every GPU loading the library holds until exit. Configs whose scratch
 * (control words, 4 copies of the M x E logits as 8-byte words, 4 copies of the
 * I fp32 intermediate values of each of the S*M + k*M (expert, row) pairs, one
 * flag per SM) exceeds it, and configs with w2_layout MOE_W2_I_H (the split-K
 * kernel's partial sums need grid x grid blocks), return MOE_ERR_UNSUPPORTED
 * before any device work. The first call on a device
 * sets the array up (resolves its device address and fills it, a blocking
 * memset). The array's address is looked up again on every call; a call that
 * finds it moved (the module was reloaded, as after cudaDeviceReset) sets the new
 * array up the same way. Every call shares the array and it keeps the last call's
 * contents; calls that overlap on the GPU (from different streams or threads, on
 * one device) race, so issue them one after another.
 *
 * Blocking: the call waits for the step on `stream` and returns its device
 * status (MOE_OK or MOE_ERR_DEVICE_TIMEOUT), as moe_decode_run_host does. So it
 * must never be made on a stream that is being captured into a CUDA graph: such
 * a call returns MOE_ERR_INVALID_ARG before any device work. MOE_ERR_UNSUPPORTED
 * also when one CTA of the launch does not fit an SM.
 * Never calls cudaMalloc, cudaFree or any allocating library routine.
 */
#define MOE_DECODE_STATIC_SCRATCH_BYTES (4u << 20)
moe_status moe_decode_run_static(const moe_decode_config* cfg, const moe_decode_weights* w, const void* x,
                                 const void* residual, void* out, int32_t m_rows, int32_t* topk_idx,
                                 float* topk_w, moe_stream_t stream);

/* Frees the handle's scratch (waits for the device first). NULL is a no-op. */
moe_status moe_decode_destroy(moe_decode_handle* h);

/* Static text for a status code. */
const char* moe_decode_status_string(moe_status s);

/* MOE_DECODE_ABI_VERSION of the loaded library. */
int32_t moe_decode_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_DECODE_H */
