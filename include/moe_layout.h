/*
 * moe_layout.h - C ABI of libmoe_layout.so: MoE expert-parallel token dispatch
 * and combine on one GPU, with the EP ranks as logical partitions of one
 * device allocation.
 *
 * Sources, cited by page title and section:
 *   "How GPUs Talk to Each Other During LLM Inference", section 7 "Expert
 *     Parallelism": dispatch sends each token's hidden state to the ranks of its
 *     top-k experts, grouped by expert; combine weights each expert output by
 *     its router score and sums the k outputs at the token's home rank.
 *   Perplexity, "Efficient and portable mixture-of-experts communication",
 *     sections "Portable kernels", "Dispatch", "Combine": count + 1 signals,
 *     private per-(expert, sender) receive regions sized by max_m, token index
 *     kept for combine, weighted sum at the receiver into a caller tensor.
 *   "NVSHMEM and DeepEP: GPU-initiated communication", sections
 *     "High-throughput mode" (FP8 dispatch with one fp32 scale per 128
 *     elements, BF16 combine) and "Low-latency mode: fixed slots, no CPU sync"
 *     (max_m slots per local expert and source rank; no host sync; static
 *     shapes).
 *
 * Conventions for every call:
 *   - Sizes: R = num_ranks logical EP ranks, T = tokens_per_rank, H = hidden,
 *     E = num_experts, L = E / R local experts, k = topk, max_m = slots per
 *     (expert, source rank). Expert e lives on rank e / L.
 *   - Slot ids: region r = e * R + src, slot s = r * max_m + pos. Rank d owns
 *     the contiguous slot range [d*L*R*max_m, (d+1)*L*R*max_m), i.e. the
 *     receiver's [local expert][source rank][max_m] buffer, ranks concatenated.
 *   - Pointers are device pointers unless stated; the caller allocates every
 *     buffer (moe_buffer_sizes gives the sizes) and the library allocates
 *     nothing and keeps no state between calls.
 *   - The step's inputs (topk_idx, x, x_scales, topk_weights) and its output
 *     (out) may instead be pinned host memory (cudaHostAlloc or
 *     cudaHostRegister, with unified addressing): the kernels then read and
 *     write them directly over the CPU-GPU link, which on Grace-based systems
 *     replaces separate host<->device copies. Every other buffer must be
 *     device memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *     asynchronous on it and never synchronise with the host, except
 *     moe_get_error.
 *   - The return value reports host-side validation (MOE_EINVAL) and launch
 *     failures (MOE_ECUDA). Errors found by a kernel are latched into the
 *     caller's device word `err` (int32, first error wins) and read with
 *     moe_get_error. Kernels never trap: they skip the offending access.
 *   - One step is moe_layout -> moe_dispatch -> (the caller's experts) ->
 *     moe_combine, in stream order on one stream.
 *   - The kernels use programmatic dependent launch: each may be scheduled
 *     while the kernel before it in the stream is still running, and waits for
 *     that kernel to complete (griddepcontrol.wait) before it reads anything.
 *     So every input may be written by the kernel enqueued immediately before
 *     the call. The one exception is moe_dispatch, which starts loading x
 *     before its wait (in a step the kernel before it is moe_layout, which
 *     never writes x): x must not be written by the kernel enqueued
 *     immediately before moe_dispatch. moe_layout_dispatch reads nothing
 *     before its wait.
 */
#ifndef MOE_LAYOUT_H
#define MOE_LAYOUT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_EINVAL = -1,    /* invalid sizes, pointers or routing */
  MOE_EOVERFLOW = -2, /* more tokens for an (expert, source) than max_m slots */
  MOE_ETIMEOUT = -3,  /* a bounded wait on a count+1 flag gave up */
  MOE_ECUDA = -4,     /* a CUDA runtime call or launch failed */
  MOE_ENOMEM = -5     /* reserved for callers that size buffers from free memory */
} moe_status;

typedef enum {
  MOE_BF16 = 0,       /* rows of H bfloat16 */
  MOE_FP8_E4M3 = 1,   /* rows of H e4m3 bytes + H/128 fp32 scales */
  MOE_BF16_TO_FP8 = 2 /* the caller's rows are H bfloat16; dispatch quantises each row once to H e4m3
                         bytes + H/128 fp32 scales (scale = amax/448 of 128 contiguous elements, code =
                         nearest-even e4m3 of x/scale in fp32, saturated to +-448) and the slots hold
                         those ("NVSHMEM and DeepEP", high-throughput section: FP8 dispatch with
                         fine-grained scales) */
} moe_dtype;

/* The problem statement: tokens, routing, EP ranks and the per-rank bound. */
typedef struct {
  int32_t num_ranks;       /* R >= 1 */
  int32_t tokens_per_rank; /* 0 <= T <= max_m */
  int32_t hidden;          /* H; multiple of 8 (bf16) or of 128 (fp8, bf16-to-fp8) */
  int32_t num_experts;     /* E, a multiple of R */
  int32_t topk;            /* 1 <= k <= min(E, 16) */
  int32_t max_m;           /* slots per (expert, source rank), >= 1 */
  int32_t dtype;           /* moe_dtype of the dispatched rows */
  int32_t num_sms;         /* SMs the dispatch kernel may occupy; 0 = all */
} moe_desc;

/* Bytes of each buffer of one step, for all R logical ranks together. */
typedef struct {
  size_t recv_x;      /* [E][R][max_m] rows (2H bytes bf16, H bytes fp8) */
  size_t recv_scales; /* [E][R][max_m][H/128] float (0 for bf16) */
  size_t recv_meta;   /* [E][R][max_m] int32x4 header per slot */
  size_t counts;      /* [E][R] int32 */
  size_t flags;       /* [E][R] uint64 */
  size_t tok_slot;    /* [R][T][k] int32 */
  size_t expert_out;  /* [E][R][max_m][H] bfloat16 */
} moe_sizes;

/* Sizes of every buffer. Host-only; no GPU needed. Per slot a receiver holds a
 * row, its scales and a 16-byte header: the per-slot message of the
 * low-latency receive-buffer estimate ("NVSHMEM and DeepEP", low-latency
 * section: hidden + hidden/128*4 + 16 bytes). Returns MOE_EINVAL for an
 * invalid desc or NULL pointers. */
moe_status moe_buffer_sizes(const moe_desc *desc, moe_sizes *out);

/* Layout (the counting side of dispatch; Perplexity, "Dispatch"). For every
 * source rank src and expert e: counts[e*R+src] = number of tokens of src that
 * chose e; flags[e*R+src] = counts + 1 (the 0 -> non-zero change means "count
 * arrived"); tok_slot[(src*T+t)*k+j] = the fixed slot of choice j of token t,
 * with pos = number of earlier tokens of src that chose the same expert (token
 * order, so positions are deterministic).
 *   topk_idx [R][T][k] int32 in [0, E), distinct within a token, or -1 for a
 *   masked choice (no expert: tok_slot = -1, nothing is sent for it and combine
 *   takes it as a zero term; no error) (read).
 *   counts [E][R] int32, flags [E][R] uint64, tok_slot [R][T][k] int32 (written).
 *   err: device int32 error word.
 * Device errors: any other expert id outside [0, E), or one repeated within a
 * token -> MOE_EINVAL and tok_slot = -1 for that entry; pos >= max_m ->
 * MOE_EOVERFLOW and tok_slot = -1. */
moe_status moe_layout(const moe_desc *desc, const int32_t *topk_idx, int32_t *counts, uint64_t *flags,
                      int32_t *tok_slot, int32_t *err, void *stream);

/* Dispatch (pack and scatter; Perplexity, "Dispatch"; "NVSHMEM and DeepEP",
 * low-latency section). Waits, bounded, until the count+1 flag of each
 * destination region is non-zero, then copies row (src, t) and its scales into
 * each of its k slots and writes the slot header {src, t, e, j}.
 *   x [R][T] rows: H bf16 (2H bytes; also for MOE_BF16_TO_FP8) or H e4m3 bytes;
 *   16-byte aligned (read).
 *   x_scales [R][T][H/128] float (MOE_FP8_E4M3 only; NULL otherwise) (read).
 *   tok_slot, flags: from moe_layout (read).
 *   recv_x [E][R][max_m] dispatched rows (2H bytes bf16, H bytes otherwise),
 *   16-byte aligned; recv_scales [E][R][max_m][H/128] (NULL for bf16);
 *   recv_meta [E][R][max_m][4] int32, 16-byte
 *   aligned (written; only slots pos < count are touched).
 * Device errors: a flag still zero after the bounded wait -> MOE_ETIMEOUT;
 * tok_slot out of range -> MOE_EINVAL; the affected copies are skipped.
 * x is loaded before the dependency wait (its loads overlap moe_layout's
 * tail), so it must not be written by the kernel enqueued immediately before
 * this call; x_scales and the rest are read after the wait. */
moe_status moe_dispatch(const moe_desc *desc, const void *x, const float *x_scales, const int32_t *tok_slot,
                        const uint64_t *flags, void *recv_x, float *recv_scales, int32_t *recv_meta,
                        int32_t *err, void *stream);

/* Layout and dispatch in one call: the same outputs as moe_layout followed by
 * moe_dispatch (same arguments, same device errors except that no flag wait
 * can time out). For decode-sized batches (T <= 1024 tokens per rank, input
 * rows of at most 16 KiB) it runs as one kernel in which every CTA computes
 * the token-order slots of its row itself, from its rank's routing, while the
 * row's loads are in flight (Perplexity, "Dispatch": the counting warp beside
 * the packing warps); otherwise it launches the two kernels. Reads nothing
 * before its dependency wait, so x, x_scales and topk_idx may come from the
 * kernel enqueued immediately before it. */
moe_status moe_layout_dispatch(const moe_desc *desc, const int32_t *topk_idx, const void *x, const float *x_scales,
                               int32_t *counts, uint64_t *flags, int32_t *tok_slot, void *recv_x,
                               float *recv_scales, int32_t *recv_meta, int32_t *err, void *stream);

/* Number of kernels one moe_layout_dispatch call launches for this desc (1 or
 * 2; an empty batch launches only the layout kernel), or MOE_EINVAL.
 * Host-only. */
int32_t moe_layout_dispatch_kernels(const moe_desc *desc);

/* Receive side of dispatch, the "hook" run when the experts want their inputs
 * (Perplexity, "Dispatch": wait for every count, then copy the payloads into
 * contiguous per-expert buffers for the grouped GEMM, keeping source rank,
 * expert and token for combine; "NVSHMEM and DeepEP", low-latency section:
 * receiving is a separate step after a send that only issued its writes).
 * Waits, bounded, for every region's count + 1 flag, checks flag - 1 == count,
 * then packs the filled slots in (expert, source rank, position) order:
 *   region_offsets[r] = filled slots of the regions before r (r = e*R + src),
 *   region_offsets[E*R] = total, so expert e's rows are
 *   [region_offsets[e*R], region_offsets[(e+1)*R]); slot s lands at packed row
 *   region_offsets[s / max_m] + s % max_m.
 *   counts, flags, recv_x, recv_scales, recv_meta, tok_slot: from layout and
 *   dispatch (read).
 *   region_offsets [E*R + 1] int32 (written).
 *   packed_x [R*T*k] dispatched rows, 16-byte aligned; packed_scales
 *   [R*T*k][H/128] (NULL for bf16); packed_meta [R*T*k][4] int32, 16-byte aligned
 *   (written: the first region_offsets[E*R] rows).
 *   tok_packed [R][T][k] int32 (written): the packed row of choice j of token t
 *   of rank src, the map moe_combine_packed gathers through; -1 for a choice
 *   with no slot (masked, or rejected by layout).
 * Device errors: a flag still zero after the bounded wait -> MOE_ETIMEOUT; a flag
 * that disagrees with its count -> MOE_EINVAL; a count above max_m ->
 * MOE_EOVERFLOW (clamped, so nothing is written out of bounds). */
moe_status moe_dispatch_recv(const moe_desc *desc, const int32_t *counts, const uint64_t *flags, const void *recv_x,
                             const float *recv_scales, const int32_t *recv_meta, const int32_t *tok_slot,
                             int32_t *region_offsets, void *packed_x, float *packed_scales, int32_t *packed_meta,
                             int32_t *tok_packed, int32_t *err, void *stream);

/* Combine reading the expert outputs in the packed layout of moe_dispatch_recv:
 * the same result as moe_combine, with choice j of token t of rank src read from
 * row tok_packed[src][t][j] of packed_y [R*T*k][H] bf16 (16-byte aligned).
 * Clears the flags like moe_combine. */
moe_status moe_combine_packed(const moe_desc *desc, const uint16_t *packed_y, const int32_t *tok_packed,
                              const float *topk_weights, uint64_t *flags, uint16_t *out, int32_t *err, void *stream);

/* Cross-node traffic of a routing ("NVSHMEM and DeepEP", high-throughput
 * section: node-limited routing and per-node deduplication). With ranks grouped
 * ranks_per_node to a node, for every source rank src:
 *   stats[src*4 + 0] = tokens T,
 *   stats[src*4 + 1] = choices whose expert's rank lies on another node (one copy per expert),
 *   stats[src*4 + 2] = distinct destination ranks on other nodes, summed over tokens (per-GPU dedup),
 *   stats[src*4 + 3] = distinct destination nodes other than its own, summed over tokens (per-node dedup).
 *   topk_idx [R][T][k] (read, device or pinned host; -1 = a masked choice, not
 *   counted); stats [R][4] int64 (written, device).
 * Device errors: an expert id outside [0, E) -> MOE_EINVAL (the choice is not counted). */
moe_status moe_route_stats(const moe_desc *desc, const int32_t *topk_idx, int32_t ranks_per_node, int64_t *stats,
                           int32_t *err, void *stream);

/* Synthetic experts for tests and benchmarks (not part of the pages' method):
 * for every filled slot (pos < counts) of an fp8 or bf16-to-fp8 step,
 * expert_out = bf16_rne(e4m3(q) * scale * (1 + e/256)), the product taken
 * exactly and rounded once. bf16 steps use identity experts: pass recv_x as
 * expert_out to moe_combine instead (this call returns MOE_EINVAL for bf16).
 *   recv_x, recv_scales, counts (read); expert_out [E][R][max_m][H] bf16,
 *   16-byte aligned (written for filled slots only). */
moe_status moe_expert_stub(const moe_desc *desc, const void *recv_x, const float *recv_scales,
                           const int32_t *counts, uint16_t *expert_out, int32_t *err, void *stream);

/* Expert stage, linear 1 with SwiGLU ("How GPUs Talk to Each Other During LLM
 * Inference", section 7, Mega MoE: between dispatch and combine each expert runs
 * linear 1, SwiGLU and linear 2; Perplexity, "Dispatch": the packed rows feed a
 * grouped GEMM). For every packed row p of expert e, i.e. region_offsets[e*R]
 * <= p < region_offsets[(e+1)*R]:
 *   h[p][i] = bf16_rne( silu(g) * u ),  silu(g) = g / (1 + exp(-g)),
 *   g = sum_c x[p][c] w_gate[e][i][c],  u = sum_c x[p][c] w_up[e][i][c],
 * bf16 products accumulated in fp32 on the tensor cores, silu in fp32.
 *   desc: dtype MOE_BF16, hidden H a multiple of 128; inter I a multiple of 128.
 *   region_offsets [E*R + 1] int32 (read; as moe_dispatch_recv writes them).
 *   packed_x [R*T*k][H] bf16 (read); w_gate, w_up [E][I][H] bf16 (read);
 *   h [R*T*k][I] bf16 (written for packed rows only). All four 16-byte aligned.
 * Host errors: MOE_EINVAL for another dtype, sizes or alignment, or more experts
 * than fit in shared memory (about 2700); MOE_ECUDA when no TMA tensor map can
 * be made. Device errors: an expert whose offsets are not a range inside
 * [0, R*T*k] -> MOE_EINVAL (its rows are skipped); a stalled pipeline ->
 * MOE_ETIMEOUT. */
moe_status moe_expert_gate_up(const moe_desc *desc, int32_t inter, const int32_t *region_offsets,
                              const void *packed_x, const void *w_gate, const void *w_up, void *h, int32_t *err,
                              void *stream);

/* Expert stage, linear 2 (same passages): for every packed row p of expert e,
 *   packed_y[p][j] = bf16_rne( sum_i h[p][i] w_down[e][j][i] ),
 * fp32 accumulation on the tensor cores. packed_y is what moe_combine_packed
 * reads.
 *   h [R*T*k][I] bf16 (read); w_down [E][H][I] bf16 (read); packed_y [R*T*k][H]
 *   bf16 (written for packed rows only). Sizes, alignment and errors as
 *   moe_expert_gate_up. */
moe_status moe_expert_down(const moe_desc *desc, int32_t inter, const int32_t *region_offsets, const void *h,
                           const void *w_down, void *packed_y, int32_t *err, void *stream);

/* Expert stage on fp8 rows, linear 1 with SwiGLU (the passages of
 * moe_expert_gate_up; "NVSHMEM and DeepEP", high-throughput section, for rows
 * sent as FP8 with one fp32 scale per 128 elements). A row's value is its e4m3
 * code times its block scale; weights are e4m3 codes with one fp32 scale per
 * 128 x 128 block. For every packed row p of expert e:
 *   hv[p][i] = silu(g) * u,  g = sum_c x[p][c] w_gate[e][i][c],  u alike,
 * fp32 accumulation on the tensor cores (code products per 128-wide K block,
 * then times the two scales); then per 128 contiguous i, in fp32:
 *   h_scales[p][i/128] = amax / 448 (1 for an all-zero block),
 *   h[p][i] = e4m3(hv / scale), round to nearest even, saturating at 448.
 *   desc: dtype MOE_FP8_E4M3 or MOE_BF16_TO_FP8 (the packed rows are e4m3),
 *   H a multiple of 128; inter I a multiple of 128.
 *   packed_x [R*T*k][H] e4m3 and packed_scales [R*T*k][H/128] f32 (as
 *   moe_dispatch_recv writes them); w_gate, w_up [E][I][H] e4m3 with
 *   w_gate_scales, w_up_scales [E][I/128][H/128] f32; h [R*T*k][I] e4m3 and
 *   h_scales [R*T*k][I/128] f32 (written for packed rows only). Row and weight
 *   pointers 16-byte aligned, scale pointers 4-byte aligned.
 * Errors as moe_expert_gate_up (MOE_EINVAL for bf16 rows). */
moe_status moe_expert_gate_up_fp8(const moe_desc *desc, int32_t inter, const int32_t *region_offsets,
                                  const void *packed_x, const float *packed_scales, const void *w_gate,
                                  const float *w_gate_scales, const void *w_up, const float *w_up_scales, void *h,
                                  float *h_scales, int32_t *err, void *stream);

/* Expert stage on fp8 rows, linear 2: for every packed row p of expert e,
 *   packed_y[p][j] = bf16_rne( sum_i h[p][i] w_down[e][j][i] ),
 * with h as moe_expert_gate_up_fp8 writes it and w_down [E][H][I] e4m3 with
 * w_down_scales [E][H/128][I/128] f32; fp32 accumulation on the tensor cores.
 * packed_y [R*T*k][H] bf16 is what moe_combine_packed reads. Sizes, alignment
 * and errors as moe_expert_gate_up_fp8. */
moe_status moe_expert_down_fp8(const moe_desc *desc, int32_t inter, const int32_t *region_offsets, const void *h,
                               const float *h_scales, const void *w_down, const float *w_down_scales,
                               void *packed_y, int32_t *err, void *stream);

/* The expert stage (moe_expert_gate_up then moe_expert_down) in one call that
 * allocates nothing. The pages have no counterpart of this call: it exists for
 * callers that may not allocate device memory. h is kept in a fixed device array
 * of the library (32 MiB), so R*T*k * inter * 2 bytes may not exceed 32 MiB
 * (MOE_ENOMEM otherwise, nothing launched). The array is shared by all calls on
 * a device: calls whose work overlaps in time race on it. Its address is asked
 * of the CUDA runtime on every call (valid in whatever context is current); the
 * first call in a context loads the library's module, so make it before any
 * stream capture. Arguments, results and other errors as moe_expert_gate_up
 * and moe_expert_down; MOE_ECUDA if the array's address cannot be obtained. */
moe_status moe_expert_mlp_noalloc(const moe_desc *desc, int32_t inter, const int32_t *region_offsets,
                                  const void *packed_x, const void *w_gate, const void *w_up, const void *w_down,
                                  void *packed_y, int32_t *err, void *stream);

/* The fp8 expert stage (moe_expert_gate_up_fp8 then moe_expert_down_fp8) in one
 * call that allocates nothing, like moe_expert_mlp_noalloc and in the same fixed
 * array: h (R*T*k * inter e4m3 bytes, rounded up to 256) and then its scales
 * (R*T*k * inter/128 floats) may not exceed 32 MiB together (MOE_ENOMEM
 * otherwise, nothing launched). The same race rule applies. Arguments, results
 * and other errors as moe_expert_gate_up_fp8 and moe_expert_down_fp8 (inter a
 * multiple of 128); MOE_ECUDA if the array's address cannot be obtained. */
moe_status moe_expert_mlp_noalloc_fp8(const moe_desc *desc, int32_t inter, const int32_t *region_offsets,
                                      const void *packed_x, const float *packed_scales, const void *w_gate,
                                      const float *w_gate_scales, const void *w_up, const float *w_up_scales,
                                      const void *w_down, const float *w_down_scales, void *packed_y, int32_t *err,
                                      void *stream);

/* Combine (Perplexity, "Combine"; "How GPUs Talk", section 7). For every token:
 * out[src][t][h] = bf16_rne( sum_{j<k} w[src][t][j] * Y[tok_slot[src][t][j]][h] ),
 * the products and sum in fp32, choices in order j = 0..k-1, weights applied at
 * the receiver. Then clears flags to zero so the next step's layout signals
 * afresh (the dispatch -> combine barrier becomes stream order).
 *   expert_out Y [E][R][max_m][H] bf16, 16-byte aligned (read at slots only).
 *   topk_weights [R][T][k] float; tok_slot [R][T][k] (read).
 *   flags [E][R] (zeroed). out [R][T][H] bf16, 16-byte aligned (written).
 * Device errors: tok_slot >= E*R*max_m -> MOE_EINVAL (the term is skipped);
 * tok_slot < 0 (an entry layout rejected) contributes nothing. */
moe_status moe_combine(const moe_desc *desc, const uint16_t *expert_out, const float *topk_weights,
                       const int32_t *tok_slot, uint64_t *flags, uint16_t *out, int32_t *err, void *stream);

/* Clear flags [E][R] and the error word (for the first step, or after an
 * aborted one). */
moe_status moe_reset(const moe_desc *desc, uint64_t *flags, int32_t *err, void *stream);

/* ---------------------------------------------------------------------------
 * Partitioned slot buffers: the receive side split the way the GPUs of an EP
 * group hold it (Perplexity, "NVSHMEM": each rank owns its private receive
 * buffers and a sender puts its rows there, then signals; "Combine": the
 * receiver's results are read back per token). With G parts (G divides R,
 * 1 <= G <= MOE_MAX_PARTS), part g holds the regions of ranks
 * [g*R/G, (g+1)*R/G): its recv_x, recv_scales, recv_meta and expert_out hold
 * global slots [g*P, (g+1)*P) at local slot s - g*P, with P = E*R*max_m / G,
 * and its flags hold regions [g*E*R/G, (g+1)*E*R/G) likewise; each buffer is
 * 1/G of the size moe_buffer_sizes gives. Slot ids (tok_slot, the slot
 * headers) and counts [E][R] stay global. The parts may be separate
 * allocations; every part is written with plain stores only.
 * --------------------------------------------------------------------------- */
#define MOE_MAX_PARTS 8

typedef struct {
  int32_t num_parts;                     /* G */
  void *recv_x[MOE_MAX_PARTS];           /* 16-byte aligned */
  float *recv_scales[MOE_MAX_PARTS];     /* NULL for bf16 rows; 4-byte aligned */
  int32_t *recv_meta[MOE_MAX_PARTS];     /* 16-byte aligned */
  uint64_t *flags[MOE_MAX_PARTS];        /* 8-byte aligned */
  void *expert_out[MOE_MAX_PARTS];       /* bf16 rows of H, 16-byte aligned; NULL where not used */
} moe_parts;

/* moe_layout_dispatch with the receive side in parts (see above): the same
 * results, each slot's row, scales and header in its part, each count + 1 flag
 * in its part; counts and tok_slot global. Reads nothing before its dependency
 * wait. Errors as moe_layout_dispatch; an invalid part table -> MOE_EINVAL. */
moe_status moe_layout_dispatch_parts(const moe_desc *desc, const int32_t *topk_idx, const void *x,
                                     const float *x_scales, int32_t *counts, int32_t *tok_slot,
                                     const moe_parts *parts, int32_t *err, void *stream);

/* moe_combine reading each expert output row from its part (parts->expert_out;
 * for bf16 identity experts the caller may pass the recv_x parts there) and
 * clearing every part's flags. */
moe_status moe_combine_parts(const moe_desc *desc, const moe_parts *parts, const float *topk_weights,
                             const int32_t *tok_slot, uint16_t *out, int32_t *err, void *stream);

/* moe_expert_stub over parts: reads each part's rows and scales, writes its
 * expert_out rows. Test and benchmark support, like moe_expert_stub. */
moe_status moe_expert_stub_parts(const moe_desc *desc, const moe_parts *parts, const int32_t *counts, int32_t *err,
                                 void *stream);

/* moe_reset over parts: clears every part's flags and the error word. */
moe_status moe_reset_parts(const moe_desc *desc, const moe_parts *parts, int32_t *err, void *stream);

/* Synchronise `stream`, read the device error word, clear it, and return its
 * value (MOE_OK if no kernel latched an error). Host-synchronising. */
moe_status moe_get_error(int32_t *err, void *stream);

/* Static description of a status code. */
const char *moe_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LAYOUT_H */
