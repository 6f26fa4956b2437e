/*
 * dsv4.h -- C ABI of the DeepSeek-V4 attention O-projection hot path on
 * GB300 (sm_103a).
 *
 * The path (vLLM docs, models/deepseek_v4/nvidia/ops/o_proj,
 * deep_gemm_fp8_o_proj):
 *     o --(inverse RoPE + per-128 FP8 quant)--> x, sx
 *       --(grouped wo_a, group g meets rows g*R:(g+1)*R)--> z [T, G, R] bf16
 *       --(wo_b over z.flatten(1))--> out [T, hidden] bf16
 *
 * Conventions for every entry point:
 *   - Sizes are int64_t or int.  Pointers marked "device" must be device
 *     memory of the current CUDA device (or managed memory); the caller owns
 *     every buffer.  The library never allocates, frees or synchronises in a
 *     compute call: it validates, then enqueues kernels on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream) and returns.
 *   - Every argument is checked on the host before any launch.  On a host
 *     error nothing is written and a negative dsv4_status is returned.  T == 0
 *     is valid and launches nothing.
 *   - Data-dependent faults (an out-of-range position, a pipeline wait that
 *     exceeded its limit) cannot be seen before the launch: the kernels record
 *     them in a device status word and never trap.  Read it with
 *     dsv4_device_status().
 *   - Inputs must be finite (the pages say nothing about NaN/Inf handling).
 *   - Calls on the same stream are ordered; concurrent calls on different
 *     streams that share output buffers race, as for any kernel.
 */
#ifndef DSV4_H
#define DSV4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dsv4_status {
    DSV4_OK = 0,
    DSV4_ERR_SHAPE = -1,       /* a shape assert of fused_inv_rope_fp8_quant, or a size rule below */
    DSV4_ERR_NULL = -2,        /* a required pointer is NULL                                      */
    DSV4_ERR_ALIGN = -3,       /* a base pointer is not 16-byte aligned (TMA and vector loads)    */
    DSV4_ERR_UNSUPPORTED = -4, /* not an sm_103 device, or a parameter the library does not serve */
    DSV4_ERR_WORKSPACE = -5,   /* workspace NULL or smaller than dsv4_o_proj_workspace_bytes()    */
    DSV4_ERR_CUDA = -6,        /* a CUDA runtime/driver call failed (launch error included)       */
    DSV4_ERR_TIMEOUT = -7,     /* device status: a kernel pipeline wait ran out of time           */
    DSV4_ERR_RANGE = -8        /* device status: a position outside [0, max_pos)                  */
} dsv4_status;

/*
 * Fused inverse RoPE + block-scaled FP8 quantisation.
 *
 * Follows vLLM docs, models/deepseek_v4/common/ops/fused_inv_rope_fp8_quant
 * (signature, parameter table, shape asserts, derived sizes), with
 * tma_aligned_scales=True: the SM100-family layout that
 * compute_fp8_einsum_recipe picks for cap.major >= 10 (o_proj page), which
 * includes GB300.  The rotated lanes are the last rope_dim of each head
 * (sglang deepseek_v4.py, MQALayer.forward: o[..., -qk_rope_head_dim:] with
 * inverse=True), paired GPT-J style (rotary_emb built with
 * is_neox_style=False): (a, b) = (x[nope+2i], x[nope+2i+1]) becomes
 * (a c + b s, b c - a s) with c = cache[p][i], s = cache[p][rope/2 + i].
 *
 *   o              device bf16 [T, H, head_dim] contiguous, H = n_groups*heads_per_group
 *   positions      device int64 [T], each in [0, max_pos)
 *   cos_sin_cache  device fp32 [max_pos, rope_dim] contiguous: cos || sin
 *   out_fp8        device e4m3 bytes, physical [G][T][D], D = heads_per_group*head_dim:
 *                  the page's [T, G, D] view with strides (D, T*D, 1)
 *   out_scale      device int32, physical [G][PK][T_al], PK = ceil(D/qgs/4),
 *                  T_al = T rounded up to a multiple of 4 (get_tma_aligned_size(T, 4)):
 *                  the page's [T, G, PK] view with strides (1, PK*T_al, T_al).
 *                  Block kb of row (t, g) is byte kb % 4 (little-endian) of
 *                  int32 kb / 4; the byte is e + 127 for the scale 2^e, e the
 *                  smallest integer with max(amax, 1e-4) <= 448 * 2^e.  Pad
 *                  columns [T, T_al) are not written.
 *
 * Errors: DSV4_ERR_SHAPE for a failed page assert (H != G*hpg, head_dim !=
 * nope+rope, head_dim % qgs, nope % qgs != qgs - rope, odd rope, T < 0,
 * max_pos <= 0); DSV4_ERR_UNSUPPORTED unless nope_dim = 448, rope_dim = 64,
 * quant_group_size = 128 (the only configuration the pages use);
 * DSV4_ERR_NULL / DSV4_ERR_ALIGN for pointers (all 16-byte aligned).
 * A position outside [0, max_pos) sets DSV4_ERR_RANGE in the device status
 * word; that token's rope lanes are then quantised unrotated.
 */
int dsv4_inv_rope_fp8_quant(const void* o, const int64_t* positions, const float* cos_sin_cache,
                            int64_t num_tokens, int64_t max_pos, int n_groups,
                            int heads_per_group, int nope_dim, int rope_dim,
                            int quant_group_size, void* out_fp8, int32_t* out_scale,
                            void* stream);

/*
 * Grouped wo_a projection with block-scaled FP8 operands.
 *
 * Follows vLLM docs, models/deepseek_v4/common/grouped_wo_a (group g of the
 * inverse-rotated output meets only rows g*R:(g+1)*R) and o_proj page,
 * deep_gemm_fp8_o_proj: fp8_einsum("bhr,hdr->bhd") with recipe (1, 1, 128)
 * into a bf16 z [T, G, R]; weight scales are 128 x 128 blocks (sglang
 * deepseek_v4.py, _dequant_fp8).
 *     z[t, g, n] = bf16( sum_k x[t,g,k] 2^ex[t,g,k/128] * W[g*R+n,k] 2^ew[(g*R+n)/128, k/128] )
 * accumulated in fp32 on the tensor cores.
 *
 *   x_fp8    device e4m3 physical [G][T][D]   (out_fp8 of the call above)
 *   x_scale  device int32 physical [G][PK][T_al] (out_scale of the call above)
 *   w_fp8    device e4m3 [G*R, D] row-major (wo_a.weight)
 *   w_scale  device UE8M0 raw bytes [G*R/128, D/128] row-major
 *   z        device bf16 [T, G, R] contiguous
 *
 * Errors: DSV4_ERR_SHAPE unless D and R are positive multiples of 128 and
 * T >= 0; DSV4_ERR_NULL / DSV4_ERR_ALIGN (16 bytes) for pointers.
 */
int dsv4_grouped_wo_a(const void* x_fp8, const int32_t* x_scale, int64_t num_tokens,
                      int n_groups, int group_dim, int o_lora_rank, const void* w_fp8,
                      const uint8_t* w_scale, void* z, void* stream);

/* Launch option of dsv4_grouped_wo_a_ex. */
#define DSV4_OVERLAP_PREVIOUS 1u

/*
 * dsv4_grouped_wo_a with launch options (flags = 0: exactly dsv4_grouped_wo_a).
 *
 * DSV4_OVERLAP_PREVIOUS: the kernel is launched with programmatic stream
 * serialization, so that it starts while the previous kernel on `stream`
 * still runs: its prologue and, for the shapes served by one CTA per tile
 * (the large FP8 shapes run on CTA pairs, which wait before any read), its
 * reads of w_fp8 and w_scale (the first pipeline stages into shared memory,
 * the rest of each CTA's first weight tile into L2) overlap that kernel, and
 * every read of x_fp8 / x_scale and every write of z waits until that kernel
 * has completed.  For the
 * weight-read-bound decode shapes this hides the launch and much of the
 * weight stream behind the kernel before (in a decode step, the quantiser).
 * The caller guarantees that the previous kernel on the stream does not write
 * w_fp8 or w_scale (weights loaded once and then only read).
 *
 * Errors: as dsv4_grouped_wo_a; DSV4_ERR_SHAPE for an unknown flag bit.
 */
int dsv4_grouped_wo_a_ex(const void* x_fp8, const int32_t* x_scale, int64_t num_tokens,
                         int n_groups, int group_dim, int o_lora_rank, const void* w_fp8,
                         const uint8_t* w_scale, void* z, unsigned flags, void* stream);

/* Largest token count the fused path below serves (decode sizes). */
#define DSV4_FUSED_MAX_TOKENS 64

/*
 * Inverse RoPE + FP8 quantisation fused into the grouped wo_a projection, for
 * decode sizes (num_tokens <= DSV4_FUSED_MAX_TOKENS).  The quantiser's work
 * (dsv4_inv_rope_fp8_quant: the same rotation, scale rule and e4m3 cast, bit
 * for bit) is done by producer warps of the GEMM kernel, which write the FP8
 * A tile and its scales straight into shared memory; the FP8 activation never
 * goes to device memory.  This is the fusion of the quantiser into the grouped
 * GEMM that the o_proj page's fused_inv_rope_fp8_quant -> fp8_einsum sequence
 * admits: z equals dsv4_grouped_wo_a applied to dsv4_inv_rope_fp8_quant's
 * output on the same inputs.  Each CTA quantises the A rows of its own
 * 128-column tile, so the quantiser's work is repeated once per column tile
 * (R / 128 times); at the decode sizes measured this makes the one launch
 * slower than the two separate ones, and dsv4_o_proj keeps the separate calls.
 *
 *   o, positions, cos_sin_cache, sizes: as dsv4_inv_rope_fp8_quant
 *   o_lora_rank  R, a positive multiple of 128
 *   w_fp8, w_scale, z: as dsv4_grouped_wo_a (z bf16 [T, G, R] contiguous)
 *
 * Errors: as dsv4_inv_rope_fp8_quant for the quantiser's arguments,
 * DSV4_ERR_SHAPE for R, DSV4_ERR_UNSUPPORTED when num_tokens exceeds
 * DSV4_FUSED_MAX_TOKENS or max_pos exceeds INT32_MAX (use the two separate
 * calls), DSV4_ERR_NULL / DSV4_ERR_ALIGN (16 bytes) for pointers.  An
 * out-of-range position sets DSV4_ERR_RANGE in the device status word, as in
 * the quantiser.
 */
int dsv4_inv_rope_grouped_wo_a(const void* o, const int64_t* positions,
                               const float* cos_sin_cache, int64_t num_tokens, int64_t max_pos,
                               int n_groups, int heads_per_group, int nope_dim, int rope_dim,
                               int quant_group_size, int o_lora_rank, const void* w_fp8,
                               const uint8_t* w_scale, void* z, void* stream);

/*
 * quantize=False variant of dsv4_inv_rope_fp8_quant: the bf16 inverse-rotated
 * groups (vLLM docs, grouped_wo_a, grouped_input: "The BF16 inverse-rotated
 * groups, [num_tokens, n_groups, group_dim]"; o_proj page,
 * deep_gemm_fp8_o_proj with quantize=use_fp8 false for a non-FP8 wo_a).
 *
 *   o, positions, cos_sin_cache, sizes: as dsv4_inv_rope_fp8_quant
 *   out_bf16   device bf16, physical [G][T][D] (the [T, G, D] view with strides
 *              (D, T*D, 1)); nope lanes are copied exactly, each rotated value
 *              is the fp32 rotation rounded to bf16 (nearest, ties to even).
 *
 * Errors: as dsv4_inv_rope_fp8_quant (quant_group_size is not an argument).
 */
int dsv4_inv_rope_bf16(const void* o, const int64_t* positions, const float* cos_sin_cache,
                       int64_t num_tokens, int64_t max_pos, int n_groups, int heads_per_group,
                       int nope_dim, int rope_dim, void* out_bf16, void* stream);

/*
 * Grouped wo_a with bf16 operands: the o_proj page's path for a non-FP8 wo_a,
 * torch.bmm of the [G, T, D] groups with wo_a.weight viewed [G, R, D]
 * transposed, into a bf16 z [T, G, R]; fp32 accumulation on the tensor cores
 * (tcgen05 kind::f16).
 *
 *   x_bf16   device bf16 physical [G][T][D] (out_bf16 of the call above)
 *   w_bf16   device bf16 [G*R, D] row-major
 *   z        device bf16 [T, G, R] contiguous
 *
 * Errors: DSV4_ERR_SHAPE unless D is a positive multiple of 64 and R of 128;
 * DSV4_ERR_NULL / DSV4_ERR_ALIGN (16 bytes) for pointers.
 */
int dsv4_grouped_wo_a_bf16(const void* x_bf16, int64_t num_tokens, int n_groups, int group_dim,
                           int o_lora_rank, const void* w_bf16, void* z, void* stream);

/*
 * Bytes of caller-owned scratch that dsv4_o_proj needs for these sizes.
 * Returns 0 for invalid sizes.  The workspace holds four parts, in this order,
 * each starting at the previous part's end rounded up to a multiple of 256
 * bytes (the first at offset 0):
 *   x   e4m3 codes of the quantised groups, physical [G][T][D]
 *   xs  their packed UE8M0 scales, int32 physical [G][PK][T_al]
 *   zq  e4m3 codes of the per-128 re-quantised bf16 z, [T][G*R] row-major
 *   zs  their packed UE8M0 scales, int32 physical [ceil(G*R/512)][T_al]
 *       (byte c/128 % 4 of word c/512 of token t for 128-column block c/128;
 *       when G*R/128 is not a multiple of 4 the last word's unused high
 *       bytes are unspecified)
 * After dsv4_o_proj returns and its kernels have run, these parts hold the
 * call's intermediate results (pad columns [T, T_al) of the scales are
 * unspecified); a caller may read them, e.g. to check each stage.
 */
size_t dsv4_o_proj_workspace_bytes(int64_t num_tokens, int n_groups, int heads_per_group,
                                   int head_dim, int o_lora_rank);

/*
 * The whole O-projection (o_proj page, deep_gemm_fp8_o_proj with an FP8
 * wo_b): inverse RoPE + FP8 quant of o, the grouped wo_a GEMM, the per-128
 * UE8M0 re-quantisation of the bf16 z.flatten(1) (fused into the wo_a
 * epilogue: z is rounded to bf16 first, then quantised exactly as a stored z
 * would be), and the dense wo_b GEMM
 *     out[t, h] = bf16( sum_c zq[t,c] 2^ez[t,c/128] * Wb[h,c] 2^eb[h/128, c/128] ).
 * The activation quantisation inside wo_b is not printed on the pages; this
 * is its plainest reading (the same per-128 UE8M0 rule as wo_a's input).
 * Three launches.
 *
 *   o, positions, cos_sin_cache, max_pos, sizes: as dsv4_inv_rope_fp8_quant
 *   wo_a_fp8, wo_a_scale : as dsv4_grouped_wo_a (w_fp8, w_scale)
 *   wo_b_fp8             device e4m3 [hidden, G*R] row-major
 *   wo_b_scale           device UE8M0 raw bytes [hidden/128, G*R/128]
 *   out                  device bf16 [T, hidden] contiguous
 *   workspace            device scratch of at least dsv4_o_proj_workspace_bytes()
 *                        bytes, 256-byte aligned; its contents are clobbered.
 *
 * Errors: as the two calls above, plus DSV4_ERR_SHAPE unless hidden is a
 * positive multiple of 128, DSV4_ERR_WORKSPACE if the workspace is NULL or too
 * small, DSV4_ERR_ALIGN if it is not 256-byte aligned.
 */
int dsv4_o_proj(const void* o, const int64_t* positions, const float* cos_sin_cache,
                int64_t max_pos, int64_t num_tokens, int n_groups, int heads_per_group,
                int nope_dim, int rope_dim, int quant_group_size, int o_lora_rank, int hidden,
                const void* wo_a_fp8, const uint8_t* wo_a_scale, const void* wo_b_fp8,
                const uint8_t* wo_b_scale, void* out, void* workspace, size_t workspace_bytes,
                void* stream);

/*
 * dsv4_o_proj, and in addition records four caller-created CUDA events
 * (cudaEvent_t handles) on `stream`: stage_events[0] before the quantisation
 * kernel and stage_events[1..3] after the quantisation, wo_a and wo_b kernels.
 * Elapsed times between consecutive events are the per-kernel device times of
 * the step, measured without a profiler.  stage_events == NULL behaves exactly
 * like dsv4_o_proj.  DSV4_ERR_CUDA if an event record fails.
 */
int dsv4_o_proj_with_events(const void* o, const int64_t* positions, const float* cos_sin_cache,
                            int64_t max_pos, int64_t num_tokens, int n_groups,
                            int heads_per_group, int nope_dim, int rope_dim,
                            int quant_group_size, int o_lora_rank, int hidden,
                            const void* wo_a_fp8, const uint8_t* wo_a_scale,
                            const void* wo_b_fp8, const uint8_t* wo_b_scale, void* out,
                            void* workspace, size_t workspace_bytes, void* const* stage_events,
                            void* stream);

/*
 * Size of the library's own scratch for dsv4_o_proj_static: 64 MiB, held on
 * every device that loads this library until the process exits.  It covers
 * dsv4_o_proj_workspace_bytes() up to this value, e.g. up to 812 tokens of the
 * 128-head, o_lora_rank 1024 configuration (82.5 KB per token).
 */
#define DSV4_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * dsv4_o_proj without a workspace argument and without any allocation.  The
 * pages have no counterpart to this entry point.
 *
 * For callers that cannot allocate device memory at call time: a C program or
 * plugin running inside an engine that owns all device memory through its own
 * pre-planned pool and gives the plugin no allocator, or code on a latency
 * path where cudaMalloc/cudaFree would synchronise the device and stall other
 * streams.  The scratch that dsv4_o_proj takes from the caller (the quantised
 * groups, the re-quantised z and their scales) lives instead in one file-scope
 * device array of DSV4_STATIC_SCRATCH_BYTES inside this library.  The caller
 * still passes and owns every input and output.  The call allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Arguments, layouts and errors are those of dsv4_o_proj.  In addition it
 * returns DSV4_ERR_WORKSPACE, launching nothing, when
 * dsv4_o_proj_workspace_bytes() for these sizes exceeds
 * DSV4_STATIC_SCRATCH_BYTES.
 *
 * The first call on a device looks up the device address of the array
 * (cudaGetSymbolAddress, once per device, with that device current); make
 * that first call before any stream capture.  Every call on a device uses the
 * same array, and the array keeps the last call's contents: calls that overlap
 * on the GPU (on different streams, or from different host threads without
 * ordering) race on it and must be serialised by the caller.  Nothing in the
 * array needs to start at zero: every byte a kernel reads was written earlier
 * in the same call.
 */
int dsv4_o_proj_static(const void* o, const int64_t* positions, const float* cos_sin_cache,
                       int64_t max_pos, int64_t num_tokens, int n_groups, int heads_per_group,
                       int nope_dim, int rope_dim, int quant_group_size, int o_lora_rank,
                       int hidden, const void* wo_a_fp8, const uint8_t* wo_a_scale,
                       const void* wo_b_fp8, const uint8_t* wo_b_scale, void* out,
                       void* stream);

/* DSV4_STATIC_SCRATCH_BYTES as this library was built with it (so that a
 * caller or a binding compiled separately can check its own copy). */
size_t dsv4_static_scratch_bytes(void);

/*
 * Eligibility of a layer for a pre-quantised attention output (vLLM docs,
 * o_proj page, rope_quant_unsupported_reason): an attention kernel may emit o
 * already inverse-rotated and cast to FP8 in the RopeQuant layout
 * (rope_quant_attn_out: DSV4_ROPE_QUANT_NUM_HEADS heads as
 * DSV4_ROPE_QUANT_NUM_HEADS / DSV4_ROPE_QUANT_HEADS_PER_GROUP group slots of
 * DSV4_ROPE_QUANT_HEADS_PER_GROUP heads x 512) only when the layer has exactly
 * that many local query heads, the per-tensor FP8 KV cache and an FP8 wo_a.
 *
 *   n_local_heads  query heads of the layer on this rank
 *   kv_cache_fp8   non-zero if the KV cache is per-tensor FP8 (e4m3)
 *   wo_a_fp8       non-zero if wo_a's weight is FP8 (e4m3)
 *   reason         if not NULL, receives NULL (eligible) or a static string
 *                  saying why not
 *
 * Returns DSV4_OK or DSV4_ERR_UNSUPPORTED.  Host only; no CUDA call.
 */
#define DSV4_ROPE_QUANT_NUM_HEADS 128
#define DSV4_ROPE_QUANT_HEADS_PER_GROUP 8
int dsv4_rope_quant_unsupported_reason(int n_local_heads, int kv_cache_fp8, int wo_a_fp8,
                                       const char** reason);

/*
 * Scratch bytes of dsv4_o_proj_prequant: the re-quantised z [T][G*R] e4m3 at
 * offset 0, then its packed scales int32 [ceil(G*R/512)][T_al] at the next
 * 256-byte boundary.  Returns 0 for invalid sizes.
 */
size_t dsv4_o_proj_prequant_workspace_bytes(int64_t num_tokens, int n_groups, int o_lora_rank);

/*
 * The O-projection from a pre-quantised attention output (vLLM docs, o_proj
 * page, deep_gemm_fp8_o_proj with a QuantizedActivation o): the attention
 * kernel already inverse-rotated o and cast it to FP8, one wo_a group per
 * slot with the live groups first, so only the padding slots are left out
 * (o.data[:, :n_groups], o.scale[:, :n_groups]) before the grouped wo_a,
 * the fused per-128 re-quantisation of the bf16 z and wo_b.  Two launches.
 *
 *   x_fp8    device e4m3, physical [n_slots][T][group_dim] (the [T, n_slots,
 *            group_dim] view with strides (group_dim, T*group_dim, 1))
 *   x_scale  device int32, physical [n_slots][PK][T_al], PK = ceil(group_dim/512)
 *            (the [T, n_slots, PK] view with strides (1, PK*T_al, T_al));
 *            slots >= n_groups are never read
 *   n_slots  group slots of the buffers (16 for the RopeQuant layout)
 *   n_groups live groups, <= n_slots
 *   wo_a_fp8, wo_a_scale, wo_b_fp8, wo_b_scale, out: as dsv4_o_proj
 *   workspace at least dsv4_o_proj_prequant_workspace_bytes(), 256-byte aligned
 *
 * Errors: DSV4_ERR_SHAPE unless group_dim, o_lora_rank and hidden are positive
 * multiples of 128 and 0 < n_groups <= n_slots; DSV4_ERR_NULL / DSV4_ERR_ALIGN
 * (16 bytes; the workspace 256) / DSV4_ERR_WORKSPACE as dsv4_o_proj.  Whether
 * a layer may take this path is dsv4_rope_quant_unsupported_reason()'s answer.
 */
int dsv4_o_proj_prequant(const void* x_fp8, const int32_t* x_scale, int64_t num_tokens,
                         int n_slots, int n_groups, int group_dim, int o_lora_rank, int hidden,
                         const void* wo_a_fp8, const uint8_t* wo_a_scale, const void* wo_b_fp8,
                         const uint8_t* wo_b_scale, void* out, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * One rank's share of group-split tensor parallelism (sglang deepseek_v4.py,
 * the column-parallel wo_a and row-parallel wo_b of the attention layer, with
 * attn_tp_all_reduce after wo_b; vLLM docs, o_proj page, wo_b as "a wrapper
 * that also reduce-scatters its output (DeepSeek-V4.1 GEMM-RS)").  The rank
 * owns the groups [g0, g0 + n_groups) of the layer: their heads of o, their
 * wo_a rows and the matching wo_b columns.  Because group g's z meets only
 * wo_b columns g*R .. (g+1)*R - 1 and the per-128 re-quantisation of z never
 * crosses a group, the rank's part of out is dsv4_o_proj over its own groups,
 * and out is the sum of the parts over all ranks.  This call writes that part
 * unrounded, in fp32, so that the sum rounds to bf16 once
 * (dsv4_sum_partials).
 *
 *   o              device bf16 [T, n_groups*heads_per_group, 512]: the rank's heads
 *   wo_a_fp8       device e4m3 [n_groups*R, D]: rows g0*R .. (g0+n_groups)*R - 1
 *   wo_a_scale     device UE8M0 [n_groups*R/128, D/128]
 *   wo_b_fp8       device e4m3 [hidden, n_groups*R]: columns g0*R .. of the layer's
 *                  wo_b, stored contiguously
 *   wo_b_scale     device UE8M0 [hidden/128, n_groups*R/128]
 *   out_partial    device fp32 [T, hidden]
 *   other arguments, workspace and errors: as dsv4_o_proj
 */
int dsv4_o_proj_partial(const void* o, const int64_t* positions, const float* cos_sin_cache,
                        int64_t max_pos, int64_t num_tokens, int n_groups, int heads_per_group,
                        int nope_dim, int rope_dim, int quant_group_size, int o_lora_rank,
                        int hidden, const void* wo_a_fp8, const uint8_t* wo_a_scale,
                        const void* wo_b_fp8, const uint8_t* wo_b_scale, float* out_partial,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Most partial outputs dsv4_sum_partials adds in one call. */
#define DSV4_MAX_PARTIALS 16

/*
 * out[i] = bf16(parts[0][i] + parts[1][i] + ... + parts[n-1][i]), summed in
 * fp32 in that order, rounded to nearest even: the partial outputs of
 * dsv4_o_proj_partial added into the layer's output (n > 1, all on this
 * device), or, with n = 1, the conversion of an fp32 reduce-scatter's result.
 *
 *   partials    HOST array of n device pointers, each fp32 [num_elems], 16-byte aligned
 *   n_partials  1 .. DSV4_MAX_PARTIALS
 *   out_bf16    device bf16 [num_elems], 16-byte aligned; may not overlap a partial
 *
 * Errors: DSV4_ERR_SHAPE for n out of range or num_elems < 0, DSV4_ERR_NULL,
 * DSV4_ERR_ALIGN.
 */
int dsv4_sum_partials(const float* const* partials, int n_partials, int64_t num_elems,
                      void* out_bf16, void* stream);

/* Human-readable name of a dsv4_status value (static string). */
const char* dsv4_status_string(int status);

/*
 * Reads the device status word of the current device (the first data-dependent
 * error any kernel recorded since the last clear: DSV4_ERR_RANGE or
 * DSV4_ERR_TIMEOUT, else DSV4_OK).  Synchronises `stream` first.  If `clear`
 * is non-zero the word is reset to DSV4_OK.  Returns DSV4_ERR_CUDA if the
 * read itself fails.
 */
int dsv4_device_status(void* stream, int clear);

/*
 * Diagnostics for the failure path of the kernels' pipeline waits (the pages
 * have no counterpart).  Enqueues one small kernel whose single waiting thread
 * uses the same bounded wait as the GEMM pipelines on a barrier that nothing
 * ever arrives on, with a limit of limit_us microseconds (1 .. 1,000,000)
 * instead of the pipelines' 2 s.  The wait gives up, records DSV4_ERR_TIMEOUT
 * in the device status word and the kernel returns normally: no trap, no
 * fault, the context stays usable.  Read the result with dsv4_device_status().
 * DSV4_ERR_SHAPE for a limit out of range.
 */
int dsv4_selftest_wait_timeout(int64_t limit_us, void* stream);

/* Number of kernel launches the last successful compute call on this host
 * thread enqueued (0 for T == 0).  For accounting in benchmarks. */
int dsv4_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DSV4_H */
