/*
 * moe_ffn.h -- C ABI of the GB300 (sm_103a) MoE FFN layer forward.
 *
 * One mixture-of-experts FFN layer for m tokens: router logits, softmax top-k
 * with renormalised weights, a stable permute of (token, expert) pairs by
 * expert, grouped SwiGLU experts (gate/up projection fused with
 * SiLU(gate) * up, then the down projection), and a routing-weighted
 * unpermute-reduce plus an optional shared-expert add.  The pipeline is the
 * one spelled out in spark_model/layers/moe/forward_prefill.rs
 * (MoeLayer::forward_prefill, doc comment and numbered steps 1-8); the
 * small-m GEMV arm follows the decode chain of span-02
 * engine/crates/model/src/gpu_model/forward.rs (forward_rows, "MoE" block:
 * router, glu, down for r <= 16 rows).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers of the current CUDA device,
 *     row-major and densely packed; the caller owns every buffer (weights,
 *     activations, outputs, workspace).  The library never allocates device
 *     memory and never synchronises the stream, so a call can be captured in
 *     a CUDA graph.  `stream` is a cudaStream_t (NULL = legacy default).
 *   - bf16 tensors are passed as `const void*` holding IEEE bfloat16 bits.
 *   - Calls return MOE_OK or an error status; on error nothing was launched
 *     unless the status is MOE_ERR_CUDA (a launch failed part-way).
 *   - m == 0 returns MOE_OK and launches nothing (metrale moe_v41 forward.rs,
 *     launch_n: early return at n == 0; forward_prefill: no grid.x = 0).
 *   - Results are deterministic: fixed reduction orders, no float atomics.
 *   - The workspace must be at least moe_workspace_size(layer, m) bytes and
 *     256-byte aligned.  Its first 256 bytes (the header) carry state between
 *     calls: counters that every call leaves at zero, and the device error
 *     word read (and cleared) by moe_device_status.  A layer zeroes the
 *     header itself when a call passes a workspace other than the one its
 *     previous call used; a caller that writes into those 256 bytes between
 *     two calls of one layer on the same workspace must zero them itself
 *     (cudaMemsetAsync on the call's stream).  Calls that share a workspace
 *     must be ordered on one stream.
 */
#ifndef MOE_FFN_GB300_H
#define MOE_FFN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols the shared library exports (everything else is hidden). */
#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* ---- status codes */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1 /* null/misaligned pointer, bad size, id out of range */
#define MOE_ERR_UNSUPPORTED 2 /* shape the kernels do not cover (see moe_layer_create) */
#define MOE_ERR_WORKSPACE 3   /* workspace smaller than moe_workspace_size() */
#define MOE_ERR_CUDA 4        /* a CUDA runtime/driver call or launch failed */
#define MOE_ERR_DEVICE 5      /* a kernel flagged an error (bounded wait expired, bad id) */

/* ---- weight formats */
#define MOE_WEIGHTS_BF16 0
/* e4m3 codes (uint8) with one fp32 scale per 128x128 block of each weight
 * matrix (blocks aligned at (0,0) over (out, in)); activations are quantised
 * to e4m3 with one fp32 scale per token per 128 contiguous inputs,
 * s = amax / 448, round-to-nearest-even, saturating. */
#define MOE_WEIGHTS_FP8_E4M3_B128 1
/* NVFP4 weights and activations (W4A4; span-02 gpu_model/forward.rs names an
 * "NVFP4 W4A4 block-scaled MMA MoE" and nothing more, so the format's usual
 * definition is taken): e2m1 codes (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6)
 * packed two per byte, element 2j in the low nibble of byte j; one e4m3
 * scale code per 16 contiguous inputs of a row; one fp32 scale per tensor.
 * A weight tensor is one expert's matrix.  Activations (x, and the down
 * projection's input h) are quantised per row: g = amax(row) / 2688 (1 for
 * an all-zero row); per 16-block sb = e4m3(RNE, saturating)(amax / (6 g));
 * code = e2m1(RNE, saturating)(v / (decode(sb) * g)), 0 where that scale is
 * 0.  Both arms take NVFP4 layers. */
#define MOE_WEIGHTS_NVFP4 2

/* ---- router scoring ("2. Batched topK dispatch" of forward_prefill.rs) */
/* softmax over the k picks; a router bias, if given, is added to the logits */
#define MOE_SCORING_SOFTMAX 0
/* sigmoid scores with a correction bias (the DeepSeek-V3 / MiniMax-M2
 * branch): s = sigmoid(L); the experts are chosen by s + bias, the weights
 * gather the pre-bias scores, divided by their sum when norm_topk_prob is
 * set, then multiplied by routed_scaling_factor */
#define MOE_SCORING_SIGMOID 1

/* ---- expert arms for moe_experts / moe_forward */
#define MOE_ARM_AUTO 0 /* pick by rows per expert (moe_select_arm) */
#define MOE_ARM_GEMV 1 /* small-m arm: each selected expert's weights streamed once */
#define MOE_ARM_GEMM 2 /* tcgen05/TMEM grouped GEMM arm fed by TMA */

typedef struct moe_config {
    int32_t hidden;       /* H: multiple of 128 (of 512 for fp8, of 256 for nvfp4 weights) */
    int32_t num_experts;  /* E: 1..1024 */
    int32_t top_k;        /* k: 1..min(E, 32) */
    int32_t inter;        /* I: expert intermediate size, multiple of 128 (of 512 for fp8, 256 for nvfp4) */
    int32_t shared_inter; /* 0 = no shared expert; otherwise must equal inter */
    int32_t weights;      /* MOE_WEIGHTS_BF16, MOE_WEIGHTS_FP8_E4M3_B128 or MOE_WEIGHTS_NVFP4 */
    int32_t scoring;      /* MOE_SCORING_SOFTMAX (0) or MOE_SCORING_SIGMOID */
    int32_t norm_topk_prob;      /* sigmoid scoring: 1 = renormalise the k weights to sum 1 */
    float routed_scaling_factor; /* sigmoid scoring: weight multiplier, finite and > 0 */
    /* Expert parallelism (the EP path of forward_prefill.rs: an all-reduce of
     * the bf16 [N, H] MoE output across ranks that each hold some experts,
     * the shared expert blended once, after the all-reduce).  0, 0 = this
     * layer holds all num_experts experts.  Otherwise it is one shard: it
     * holds experts [expert_begin, expert_end), 0 <= begin < end <=
     * num_experts, and its routed weight tensors are stacked over those
     * experts only (w1, w3 [end - begin, I, H] ...).  The router still
     * scores all num_experts experts (router_w [num_experts, H]) and the ids
     * stay global; a shard's moe_forward / moe_experts write the partial
     * routed sum over the pairs whose expert it holds (the other pairs are
     * dropped, not an error) and leave the shared expert out:
     * moe_shared_expert_add adds it after the caller's all-reduce. */
    int32_t expert_begin;
    int32_t expert_end;
} moe_config;

/* Stacked expert weights in nn.Linear (out, in) layout.
 *   routed:  w1, w3 [E, I, H]   w2 [E, H, I]
 *   shared:  w1, w3 [I, H]      w2 [H, I]        (E = 1 of the same layout)
 *   fp8 only: s1, s3 [E, I/128, H/128]  s2 [E, H/128, I/128]  (fp32)
 * Element type: bf16 or e4m3 codes (uint8) per moe_config.weights.
 * nvfp4: w1, w3 uint8 [E, I, H/2], w2 uint8 [E, H, I/2] (packed codes);
 *   sb1, sb3 uint8 [E, I, H/16], sb2 uint8 [E, H, I/16] (e4m3 block scales);
 *   s1, s3, s2 fp32 [E] (one scale per expert matrix; [1] for the shared
 *   expert).  sb* must be NULL for the other formats.
 * gate (shared expert only, else NULL): fp32 [H]; when set, the shared
 * expert's output is scaled per token by sigmoid(sum_h x[h] gate[h])
 * (forward_prefill.rs step "8. Blend shared expert"); NULL adds it with
 * weight 1.
 * Pointers must be 16-byte aligned.  The weights must outlive the layer. */
typedef struct moe_expert_weights {
    const void* w1;
    const void* w3;
    const void* w2;
    const float* s1;
    const float* s3;
    const float* s2;
    const float* gate;
    const uint8_t* sb1;
    const uint8_t* sb3;
    const uint8_t* sb2;
} moe_expert_weights;

typedef struct moe_layer moe_layer;

/* Create a layer handle on the current CUDA device.  The handle keeps a copy
 * of the config, the weight pointers and host-side TMA descriptors of the
 * weights; it owns no device memory.  `shared` may be NULL (and must be when
 * cfg->shared_inter == 0).  Returns MOE_ERR_UNSUPPORTED for shapes outside
 * the documented ranges. */
MOE_API int moe_layer_create(const moe_config* cfg, const moe_expert_weights* routed,
                     const moe_expert_weights* shared, moe_layer** out);
MOE_API int moe_layer_destroy(moe_layer* layer);

/* Workspace bytes a call with m tokens needs (any entry point). */
MOE_API int moe_workspace_size(const moe_layer* layer, int64_t m, size_t* bytes);

/* Which arm MOE_ARM_AUTO takes for m tokens (MOE_ARM_GEMV or MOE_ARM_GEMM). */
MOE_API int moe_select_arm(const moe_layer* layer, int64_t m);

/* Steps 1-2 of forward_prefill ("Gate GEMM", "Batched topK dispatch").
 * Softmax scoring (norm_topk_prob): logits[t,e] = sum_h x[t,h] Wr[e,h]
 * (+ bias[e]) in fp32; topk_ids[t,:] = the k largest logits in descending
 * order (equal logits: lower expert index first); topk_w[t,j] =
 * exp(L_j - L_0) / sum over the k selected of exp(L_i - L_0).
 * Sigmoid scoring: logits carry no bias; with s = sigmoid(L) (fp32),
 * topk_ids = the k largest s + bias (same order rules); topk_w[t,j] =
 * s_j (/ sum of the k s when norm_topk_prob) * routed_scaling_factor.
 *   x        bf16 [m, H]           router_w fp32 [E, H]
 *   router_bias fp32 [E] or NULL   logits_out fp32 [m, E] or NULL
 *   topk_ids int32 [m, k]          topk_w fp32 [m, k]                       */
MOE_API int moe_route(const moe_layer* layer, const void* x, int64_t m, const float* router_w,
              const float* router_bias, float* logits_out, int32_t* topk_ids, float* topk_w,
              void* workspace, size_t workspace_bytes, void* stream);

/* Step 3 of forward_prefill ("Sort tokens by expert"), as a stable counting
 * sort of the pairs p = t*k + j by expert topk_ids[p]:
 *   expert_offsets int32 [E+1]: exclusive prefix sum of per-expert counts
 *   sorted_pair    int32 [m*k]: pair at sorted slot s (ascending p within an expert)
 *   slot_of_pair   int32 [m*k]: inverse of sorted_pair
 * Ids outside [0, E) set the device error word (MOE_ERR_DEVICE).  Such a pair
 * is dropped: its slot_of_pair entry is -1, expert_offsets[E] counts only the
 * valid pairs (so it is then below m*k), and sorted_pair holds -1 from that
 * count on.  On an expert-parallel shard E is the shard's expert count
 * (expert_offsets [E+1] over its experts, in order) and pairs of the other
 * shards' experts are dropped the same way without an error.               */
MOE_API int moe_permute(const moe_layer* layer, const int32_t* topk_ids, int64_t m,
                int32_t* expert_offsets, int32_t* sorted_pair, int32_t* slot_of_pair,
                void* workspace, size_t workspace_bytes, void* stream);

/* moe_permute for callers that cannot allocate device memory at all: code
 * running while a CUDA graph is being captured, real-time serving loops that
 * forbid allocator calls after start-up, and host runtimes that own no device
 * allocator and only hold the tensors handed to them.  The pages have no
 * counterpart of this entry point; it computes exactly what moe_permute does
 * (same outputs, same kernels) but takes no workspace.
 *   topk_ids int32 [m, top_k]; expert_offsets int32 [num_experts + 1];
 *   sorted_pair, slot_of_pair int32 [m * top_k] -- as for moe_permute.
 * Its scratch is a fixed 320 KiB array inside this library's device memory
 * (each GPU that loads the library holds it until the process exits).  A
 * call whose scratch would not fit -- more than 320 KiB of per-chunk
 * histograms, about E * m * top_k / 512 bytes -- returns MOE_ERR_UNSUPPORTED
 * and launches nothing.  It calls no allocator (no cudaMalloc, cudaFree or
 * allocating library routine).
 * All calls on a device share that one array and it keeps the last call's
 * contents: each call clears the part that must start at zero itself, but two
 * calls that overlap on the GPU (different streams without ordering between
 * them) race on it; order them on one stream.  Every call looks up the
 * array's device address on the current device (a host-side query); the
 * first lookup on a device loads this library's device code there, so make
 * the first call before any stream capture begins.
 * Out-of-range ids are handled as in moe_permute (the pair is dropped,
 * slot_of_pair -1, expert_offsets[E] counts only the valid pairs, sorted_pair
 * -1 from there on), but with
 * no workspace there is no error word the caller can read: a caller that may
 * pass such ids checks expert_offsets[E] == m * top_k after the stream.     */
MOE_API int moe_permute_noalloc(const int32_t* topk_ids, int64_t m, int32_t top_k, int32_t num_experts,
                                int32_t* expert_offsets, int32_t* sorted_pair, int32_t* slot_of_pair,
                                void* stream);

/* Steps 3-8 for a given routing: permute, grouped gate/up + SiLU(gate)*up,
 * grouped down, then out[t] = sum_j topk_w[t,j] * y_{t,j} (+ shared expert
 * output, weight 1 or its sigmoid gate), accumulated in fp32 in j order and
 * stored as bf16.
 *   x bf16 [m, H]; topk_ids int32 [m, k]; topk_w fp32 [m, k]; out bf16 [m, H]
 * out is fully overwritten (metrale moe_v41 forward.rs: acc is cleared before
 * any routed or shared row is added).  arm: MOE_ARM_*.                      */
MOE_API int moe_experts(const moe_layer* layer, const void* x, int64_t m, const int32_t* topk_ids,
                const float* topk_w, void* out, int arm, void* workspace,
                size_t workspace_bytes, void* stream);

/* out[t, :] = bf16(out[t, :] + shared(x[t, :])): the shared expert alone
 * (weight 1, or its sigmoid gate), added to out in fp32 and rounded once --
 * forward_prefill.rs's "defer shared expert blend until after all-reduce",
 * the last step of an expert-parallel layer whose ranks each ran moe_forward
 * on a shard and all-reduced the partial outputs.  Works on any layer with a
 * shared expert (MOE_ERR_INVALID_ARG without one).  x bf16 [m, H]; out bf16
 * [m, H], read and written; arm as for moe_experts (AUTO: the GEMV arm up to
 * 64 tokens).  Workspace as for the other calls (moe_workspace_size covers
 * it).                                                                      */
MOE_API int moe_shared_expert_add(const moe_layer* layer, const void* x, int64_t m, void* out, int arm,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* The whole layer: moe_route then moe_experts on one stream, no host sync.
 * topk_ids_out / topk_w_out may be NULL (the routing then stays in the
 * workspace).                                                               */
MOE_API int moe_forward(const moe_layer* layer, const void* x, int64_t m, const float* router_w,
                const float* router_bias, void* out, int32_t* topk_ids_out, float* topk_w_out,
                int arm, void* workspace, size_t workspace_bytes, void* stream);

/* The whole layer with the layer tail folded into its combine (ferrum
 * qwen3_moe/forward_layer.rs: weighted_sum_residual_norm writes the weighted
 * sum into the residual stream and takes the next layer's rms_norm of the
 * result).  In place of out:
 *   residual[t,h] <- bf16(residual[t,h] + moe_out[t,h])   (moe_out: the layer
 *                    output in fp32, before moe_forward would round it)
 *   norm_out[t,h]  = bf16(r[t,h] / sqrt(sum_h r[t,h]^2 / H + eps) * norm_w[h]),
 *                    r = the new residual's values
 *   residual bf16 [m, H], in/out, aliasing neither x nor norm_out;
 *   norm_w fp32 [H]; norm_out bf16 [m, H]; eps >= 0; H <= 24576.
 * Everything else (routing outputs, arm, workspace, stream) as moe_forward. */
MOE_API int moe_forward_residual_rmsnorm(const moe_layer* layer, const void* x, int64_t m, const float* router_w,
                const float* router_bias, void* residual, const float* norm_w, float eps, void* norm_out,
                int32_t* topk_ids_out, float* topk_w_out, int arm, void* workspace, size_t workspace_bytes,
                void* stream);

/* Activation quantisation of the fp8 layers (the expert input and the down
 * projection's input): per row, per block of 128 contiguous elements,
 * s = amax / 448 (IEEE fp32 divide), code = e4m3(x / s) rounded to nearest
 * even and saturated to +-448; an all-zero block gets s = 1 and zero codes.
 *   x bf16 [rows, n]; codes uint8 [rows, n]; scales fp32 [rows, n/128];
 *   n a multiple of 128.  Needs no layer and no workspace.                  */
MOE_API int moe_act_quant_fp8(const void* x, int64_t rows, int64_t n, uint8_t* codes, float* scales,
                              void* stream);

/* Activation quantisation of the NVFP4 layers, per row as described at
 * MOE_WEIGHTS_NVFP4 (the same kernel quantises x inside moe_forward).
 *   x bf16 [rows, n]; codes uint8 [rows, n/2] (packed); block_scales uint8
 *   [rows, n/16] (e4m3 codes); row_scales fp32 [rows]; n a multiple of 16.
 * Needs no layer and no workspace.                                          */
MOE_API int moe_act_quant_nvfp4(const void* x, int64_t rows, int64_t n, uint8_t* codes, uint8_t* block_scales,
                                float* row_scales, void* stream);

/* The same quantisation of fp32 rows: the kernel that quantises the down
 * projection's input h inside moe_forward (the NVFP4 layers keep h in fp32
 * between the gate/up product and its quantisation).
 *   x fp32 [rows, n], 16-byte aligned; everything else as moe_act_quant_nvfp4.
 * Finite inputs only.                                                       */
MOE_API int moe_act_quant_nvfp4_f32(const float* x, int64_t rows, int64_t n, uint8_t* codes,
                                    uint8_t* block_scales, float* row_scales, void* stream);

/* Synchronises `stream` and reads the device error word of `workspace`: the
 * first device error of the calls made on it since the word was last read
 * (0 = none).  A set word is cleared (on `stream`) after it is read.
 * Returns MOE_OK, MOE_ERR_DEVICE when the word was set, or MOE_ERR_CUDA.    */
MOE_API int moe_device_status(void* workspace, void* stream, int32_t* device_code);

/* Router weight preparation (optional).  For m > 64 tokens (and E <= 256)
 * the router runs on the tensor cores over three bf16 planes whose sum
 * represents the fp32 router weight (hi, mid, lo); each call splits router_w
 * into its workspace first.  moe_router_prepare does that split once, into
 * `planes` (caller-owned device memory of moe_router_planes_size bytes,
 * 256-byte aligned, alive while prepared), on `stream`; later calls on this
 * layer that pass the same router_w pointer use those planes and skip the
 * split.  Only the pointer is compared: after rewriting the weight in place,
 * call moe_router_prepare again (or with router_w or planes NULL, which
 * forgets the prepared weight).  Results are identical either way.
 * (forward_prefill.rs's gate GEMM reads its router weight every call; this
 * is the load-time step an engine would run once per layer.)               */
MOE_API int moe_router_planes_size(const moe_layer* layer, size_t* bytes);
MOE_API int moe_router_prepare(moe_layer* layer, const float* router_w, void* planes, size_t planes_bytes,
                               void* stream);

/* Limit, in nanoseconds of GPU wall time, of every bounded wait inside the
 * grouped-GEMM kernels (the mbarrier waits between their TMA producer,
 * tensor-core issuer and epilogue warps); 0 restores the default of 2 s.
 * A wait that runs out makes its kernel record DEV_ERR_TIMEOUT (2) in the
 * workspace's device error word, stop issuing work, wait (2 s at most) for
 * the copies and MMAs it already issued, free its tensor memory and return;
 * that call's outputs are then unspecified and moe_device_status reports
 * MOE_ERR_DEVICE, which also clears the word.  For tests of this
 * failure path (with moe_layer_stall_test) and for callers that want a hung
 * pipeline reported sooner; it takes effect from the next call on `layer`.
 * (The failure handling of forward_prefill.rs is Rust's Result/ensure!; this
 * is its device-side counterpart.)                                           */
MOE_API int moe_layer_set_wait_limit(moe_layer* layer, uint64_t ns);

/* Test of that failure path without any fault: while enabled (1), the bf16
 * grouped-GEMM kernels of calls on `layer` make their tensor-core issuer
 * first wait on an mbarrier that no thread ever completes, so that wait runs
 * out after the wait limit and the kernel takes the abort path above (no MMA
 * is issued; the TMA copies already issued are waited for; tensor memory is
 * freed).  0 turns it off.  Other weight formats and the GEMV arm ignore it. */
MOE_API int moe_layer_stall_test(moe_layer* layer, int enable);

/* Kernels the last successful call on `layer` launched (for launch counting). */
MOE_API int moe_last_launch_count(const moe_layer* layer);

/* Optional per-kernel timing for profiling: while enabled, each kernel
 * launch of a call on `layer` is bracketed by two CUDA events on the call's
 * stream (so calls are then not capturable in a CUDA graph).  Enabling or
 * disabling resets the totals.  moe_kernel_timing_read synchronises on the
 * recorded events and returns the summed device time (ms) and launch count of
 * kernel `kernel` (0 .. moe_kernel_count()-1, named by moe_kernel_name). */
MOE_API int moe_kernel_timing_enable(moe_layer* layer, int enable);
MOE_API int moe_kernel_timing_read(moe_layer* layer, int kernel, double* total_ms, int64_t* launches);
MOE_API int moe_kernel_count(void);
MOE_API const char* moe_kernel_name(int kernel);

/* Human-readable name of a status code (static storage). */
MOE_API const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_GB300_H */
