/*
 * dit_attn.h -- C ABI of libditattn.so: blockwise DiT attention with on-chip
 * chunk merging (and its per-chunk, key-range, Torus-pipelined and
 * chunk-parallel forms), the standalone log-sum-exp merge, and the
 * classifier-free guidance combine with its fused rel-MAE, for NVIDIA B300
 * (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer is a DEVICE pointer owned by the caller (dit_attn_fwd_torus
 *    also takes pinned host sources).  The library allocates no memory on any
 *    call path; per device it keeps, in static __device__ variables, a 4-byte
 *    status word with its read-back copy and the 64.25 KiB scratch array of
 *    cfg_combine_relmae_static.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream of
 *    the current device) and return after the launch.  A status other than
 *    DIT_OK means nothing was launched, except DIT_ERR_LAUNCH.
 *  - Arguments are checked on the host before anything touches the GPU:
 *    NULL or non-16-byte-aligned pointers, non-positive or overflowing sizes
 *    and unsupported shapes are rejected with an error code and no launch.
 *  - Device-side waits are bounded (about one second).  A wait that runs out
 *    makes the kernel give up without trapping and sets the status word, which
 *    dit_last_device_status() reports as DIT_ERR_DEVICE_TIMEOUT.
 *  - The device must be compute capability 10.3 (B300); others get
 *    DIT_ERR_UNSUPPORTED_DEVICE.
 *
 * Citations name the page and the section each operation comes from; the
 * pages print no formula, so each definition is the textbook form of what the
 * section describes.
 */
#ifndef DIT_ATTN_H
#define DIT_ATTN_H

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t; callers may pass a cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *dit_stream_t;

typedef enum {
  DIT_OK = 0,
  DIT_ERR_INVALID_ARG = -1,        /* NULL pointer, bad size or count */
  DIT_ERR_UNSUPPORTED_SHAPE = -2,  /* e.g. head dimension not in {64, 72, 128} */
  DIT_ERR_MISALIGNED = -3,         /* a pointer is not 16-byte aligned */
  DIT_ERR_UNSUPPORTED_DEVICE = -4, /* not an sm_103 device */
  DIT_ERR_LAUNCH = -5,             /* the CUDA launch itself failed */
  DIT_ERR_DEVICE_TIMEOUT = -6,     /* a bounded device-side wait ran out */
  DIT_ERR_CUDA = -7                /* another CUDA runtime or driver error */
} dit_status;

/*
 * dit_attn_fwd -- full bidirectional multi-head self-attention over a DiT token
 * sequence, computed blockwise over n_kv_chunks contiguous K/V chunks whose
 * partial outputs and log-sum-exps are merged on chip.
 *
 * Source: "xDiT: an Inference Engine for DiTs with Massive Parallelism"
 * (abstract: attention over the token sequence, split by sequence
 * parallelism); "SwiftFusion: Scalable Sequence Parallelism for Distributed
 * Inference of Diffusion Transformers on GPUs" (ideas 1 and 2: ring attention
 * and Torus attention compute one piece of K/V at a time and fold each piece's
 * result into the output).  Per (b, h), with s_ij = q_i . k_j / sqrt(D):
 *     LSE_i = ln sum_j exp(s_ij),   O_i = sum_j exp(s_ij - LSE_i) v_j.
 * Chunk c covers keys [floor(c S / n), floor((c + 1) S / n)); each chunk's
 * (O_c, LSE_c) is folded into the running result by
 *     LSE = ln(exp(LSE) + exp(LSE_c)),
 *     O   = exp(LSE_old - LSE) O + exp(LSE_c - LSE) O_c,
 * so every chunk count gives the unchunked result up to rounding.
 *
 *   q, k, v   bf16 [B, H, S, D], contiguous, 16-byte aligned.
 *   out       bf16 [B, H, S, D], contiguous, 16-byte aligned; must not alias
 *             q, k or v.
 *   lse       fp32 [B, H, S] natural-log LSE of each row, or NULL.
 *   B, H, S   >= 1, with B * H <= 2^31 - 1 (element offsets are 64-bit).
 *   D         64, 72 or 128 (else DIT_ERR_UNSUPPORTED_SHAPE).
 *   n_kv_chunks  1 <= n_kv_chunks <= S (else DIT_ERR_INVALID_ARG).
 */
dit_status dit_attn_fwd(const void *q, const void *k, const void *v, void *out,
                        float *lse, int B, int H, int S, int D, int n_kv_chunks,
                        dit_stream_t stream);

/*
 * dit_attn_fwd_partials -- the per-chunk half of dit_attn_fwd: for every
 * chunk c of the same balanced partition, writes the chunk's normalised
 * partial output O_c and its LSE_c without merging.  This is what each device
 * of a ring / Torus sequence-parallel split holds before the recombination
 * ("SwiftFusion ...", ideas 1 and 2); dit_attn_merge then recombines them.
 *
 *   q, k, v    as for dit_attn_fwd.
 *   partials   fp32 [n_kv_chunks, B * H * S, D], 16-byte aligned.
 *   lses       fp32 [n_kv_chunks, B * H * S], 16-byte aligned.
 *   Other arguments and errors as for dit_attn_fwd.
 */
dit_status dit_attn_fwd_partials(const void *q, const void *k, const void *v,
                                 float *partials, float *lses, int B, int H,
                                 int S, int D, int n_kv_chunks,
                                 dit_stream_t stream);

/*
 * dit_attn_fwd_split -- dit_attn_fwd computed chunk-parallel: one CTA per
 * (query-tile pair, chunk c of the balanced partition into n_split chunks)
 * writes the chunk's normalised fp32 partial O_c and LSE_c to the caller's
 * workspace (dit_attn_fwd_partials), then a second kernel merges the chunks
 * of every row by their log-sum-exp weights and writes out (bf16) and lse.
 * It serves launches with few (batch, head, query-tile pair) units, such as
 * one device's share of the heads under a head-parallel split, where the
 * merged launch leaves SMs idle: each chunk adds a CTA per pair.  Source:
 * "xDiT: an Inference Engine for DiTs with Massive Parallelism" (abstract:
 * sequence parallelism splits the attention of a long token sequence);
 * "SwiftFusion ..." (ideas 1 and 2: every piece of K/V yields a partial
 * result, folded in by its log-sum-exp).  Same result as dit_attn_fwd with
 * n_kv_chunks = n_split, up to rounding.
 *
 *   q, k, v, out, lse, B, H, S, D   as for dit_attn_fwd.
 *   n_split    1 <= n_split <= S (else DIT_ERR_INVALID_ARG); the partials
 *              must fit the merge's limits (B * H * S * D < 2^40 and
 *              n_split * B * H * S * D <= 2^46).
 *   workspace  device memory of at least
 *              dit_attn_split_workspace_bytes(B, H, S, D, n_split) bytes,
 *              16-byte aligned, overlapping no other buffer of the call;
 *              owned by the caller, reusable by later calls on the same
 *              stream (nothing in it needs clearing).  Calls that share one
 *              workspace must not overlap on the GPU.
 *   workspace_bytes  its size (too small: DIT_ERR_INVALID_ARG).
 * Launches the partials kernel, then the merge kernel as a programmatic
 * dependent launch on the same stream (it may start while the first kernel's
 * last CTAs run and waits for all of them before reading the workspace).
 */
dit_status dit_attn_fwd_split(const void *q, const void *k, const void *v,
                              void *out, float *lse, int B, int H, int S, int D,
                              int n_split, void *workspace,
                              size_t workspace_bytes, dit_stream_t stream);

/*
 * dit_attn_split_workspace_bytes -- the workspace dit_attn_fwd_split needs:
 * fp32 partials [n_split, B * H * S, D] followed, from the next 256-byte
 * boundary, by their LSEs [n_split, B * H * S], padded to 256 bytes.
 * Returns 0 for invalid sizes (those dit_attn_fwd_split rejects) or an
 * unsupported D.
 */
size_t dit_attn_split_workspace_bytes(int B, int H, int S, int D, int n_split);

/*
 * dit_attn_fwd_range -- attention of every query over one key range
 * [j0, j1): the computation a device of a ring / Torus sequence-parallel
 * split performs on the piece of K/V it holds ("SwiftFusion ...", ideas 1 and
 * 2: each piece is computed as it arrives and its partial result folded in
 * later).  Per (b, h) and query row i, with s_ij = q_i . k_j / sqrt(D):
 *     LSE_i = ln sum_{j0 <= j < j1} exp(s_ij),
 *     out_i = sum_{j0 <= j < j1} exp(s_ij - LSE_i) v_j.
 *
 *   q, k, v      bf16 [B, H, S, D] as for dit_attn_fwd.  Only key rows
 *                [j0, j1) of k and v are read; the other rows may hold
 *                anything (NaN included) or still be in flight.
 *   out          fp32 [B * H * S, D], 16-byte aligned.
 *   lse          fp32 [B * H * S], 16-byte aligned.
 *   j0, j1       0 <= j0 < j1 <= S (else DIT_ERR_INVALID_ARG).
 */
dit_status dit_attn_fwd_range(const void *q, const void *k, const void *v,
                              float *out, float *lse, int B, int H, int S,
                              int D, int j0, int j1, dit_stream_t stream);

/*
 * dit_attn_fwd_torus -- Torus-style chunked attention on one GPU: the K/V
 * rows of chunk c (the balanced partition of dit_attn_fwd) are copied from
 * k_src / v_src into k / v on copy_stream, one event per chunk, and chunk c
 * is computed on stream (dit_attn_fwd_range into partials[c], lses[c]) as
 * soon as its own rows have arrived, while later chunks are still being
 * copied; then
 * dit_attn_merge combines the partials into out / lse_out.  Source:
 * "SwiftFusion ..." (idea 2: Torus attention splits a received block into
 * pieces and computes piece i while piece i + 1 arrives); on one GPU the
 * arrival is a copy and the overlap is between the copy engine and the SMs.
 *
 *   q            bf16 [B, H, S, D] device.
 *   k_src, v_src bf16 [B, H, S, D]: pinned host or device memory.
 *   k, v         bf16 [B, H, S, D] device buffers the copies land in.
 *   partials     fp32 [n_kv_chunks, B * H * S, D]; lses fp32 [n_kv_chunks, B * H * S].
 *   out          fp32 [B * H * S, D]; lse_out fp32 [B * H * S] or NULL.
 *   n_kv_chunks  1 <= n_kv_chunks <= min(S, 64).
 *   copy_stream  the stream of the copies (NULL or == stream: no overlap).
 * The copies wait for the work queued on `stream` before this call; the
 * result is complete when `stream` reaches the end of this call's work.
 * Uses per-device events created on the first call (no device memory).
 */
dit_status dit_attn_fwd_torus(const void *q, const void *k_src,
                              const void *v_src, void *k, void *v,
                              float *partials, float *lses, float *out,
                              float *lse_out, int B, int H, int S, int D,
                              int n_kv_chunks, dit_stream_t stream,
                              dit_stream_t copy_stream);

/*
 * dit_attn_merge -- log-sum-exp merge of n partial attention results, the
 * recombination step of ring / Torus sequence-parallel attention
 * ("SwiftFusion ...", ideas 1 and 2).  For each row r:
 *     M = max_c LSE_c[r],  LSE[r] = M + ln sum_c exp(LSE_c[r] - M),
 *     out[r] = sum_c exp(LSE_c[r] - LSE[r]) O_c[r].
 * A partial with LSE_c[r] = -inf has weight 0 and is not read; a row whose
 * partials are all -inf gives out = 0, LSE = -inf.
 *
 *   partials  fp32 [n, rows, D], contiguous, 16-byte aligned.
 *   lses      fp32 [n, rows], contiguous, 16-byte aligned.
 *   n         >= 1.
 *   out       fp32 [rows, D], 16-byte aligned; must not alias the inputs.
 *   lse_out   fp32 [rows], or NULL.
 *   rows      >= 1; D >= 1.
 */
dit_status dit_attn_merge(const float *partials, const float *lses, int n,
                          float *out, float *lse_out, long long rows, int D,
                          dit_stream_t stream);

/*
 * cfg_combine -- classifier-free guidance combine of the conditional and the
 * unconditional noise predictions, out = eps_u + w (eps_c - eps_u),
 * elementwise.  Source: "Accelerating Diffusion via Hybrid Data-Pipeline
 * Parallelism Based on Conditional Guidance Scheduling" (Technische
 * Zusammenfassung 2A: one path with the prompt c, one with c = empty, joined
 * after each denoising step); "xDiT ..." (abstract: CFG parallelism).
 *
 *   eps_c, eps_u, out  fp32 [numel], 16-byte aligned; out may alias eps_c
 *                      or eps_u (the operation is elementwise).
 *   numel              >= 1.
 */
dit_status cfg_combine(const float *eps_c, const float *eps_u, float w,
                       float *out, long long numel, dit_stream_t stream);

/*
 * cfg_combine_relmae -- cfg_combine fused with the discrepancy between the two
 * guidance paths, measured in the same pass.  Source: "Accelerating Diffusion
 * via Hybrid Data-Pipeline Parallelism Based on Conditional Guidance
 * Scheduling" (Technische Zusammenfassung 2B: the switch points between its
 * three phases are chosen from the rel-MAE between the conditional and the
 * unconditional noise; the page gives no formula, the reading taken is
 * sum |eps_c - eps_u| / sum |eps_u|).
 *
 *   eps_c, eps_u, out, numel, w   as for cfg_combine (out may alias an input).
 *   sums   fp64 [3] device, 8-byte aligned, not overlapping the other buffers:
 *          set to {sum |eps_c - eps_u|, sum |eps_u|, rel-MAE} with
 *          rel-MAE = sums[0] / sums[1], computed on the device; an all-zero
 *          eps_u gives 0 when eps_c == eps_u everywhere and +inf otherwise.
 *          This call zeroes the three values before its kernel runs; while
 *          the kernel runs, sums[2] holds its count of finished blocks.  The
 *          sums are accumulated in fp32 per thread and fp64 beyond, in an
 *          order that may vary between calls in the last bits.
 */
dit_status cfg_combine_relmae(const float *eps_c, const float *eps_u, float w,
                              float *out, long long numel, double *sums,
                              dit_stream_t stream);

/* Largest numel cfg_combine_relmae_static accepts (2^28 elements). */
#define DIT_RELMAE_STATIC_MAX_NUMEL (1LL << 28)

/*
 * cfg_combine_relmae_static -- cfg_combine_relmae with nothing asked of the
 * caller beyond its output and nothing allocated: the per-block partial sums
 * live in a fixed array of this library in device memory (64.25 KiB per
 * device, found with cudaGetSymbolAddress on the first call on each device),
 * and the last block adds them in block order, so repeated calls on the same
 * inputs give the same bits.  The pages have no counterpart to this entry
 * point: the fixed scratch array is this library's choice (the rel-MAE itself
 * follows the Hybridiff page, section 2B, as for cfg_combine_relmae).
 *
 *   eps_c, eps_u, w, out, sums   as for cfg_combine_relmae; sums is written
 *          (not accumulated): {sum |eps_c - eps_u|, sum |eps_u|, rel-MAE}.
 *   numel  1 <= numel <= DIT_RELMAE_STATIC_MAX_NUMEL, else
 *          DIT_ERR_INVALID_ARG (each block of 256 threads owns a slab of
 *          65536 elements and the array holds 4096 slabs).
 * The call clears the array's block counter (cudaMemsetAsync on `stream`)
 * before its kernel.  The array is shared by every call on a device: two
 * calls whose kernels overlap on one device (other streams, other host
 * threads) race on it and give wrong sums; serialise them.
 */
dit_status cfg_combine_relmae_static(const float *eps_c, const float *eps_u,
                                     float w, float *out, long long numel,
                                     double *sums, dit_stream_t stream);

/*
 * dit_last_device_status -- after the work queued on `stream`, reads and
 * clears this device's status word in one atomic exchange (a one-thread
 * kernel on `stream`), then synchronises `stream`.  Returns
 * DIT_ERR_DEVICE_TIMEOUT if a kernel gave up on a bounded wait since the last
 * call, DIT_ERR_CUDA if the copy or the synchronisation failed, else DIT_OK.
 * A timeout recorded by a kernel on another stream after the exchange stays
 * in the word for the next call.
 */
dit_status dit_last_device_status(dit_stream_t stream);

/*
 * dit_selftest_bounded_wait -- exercises the failure path of the bounded
 * device-side waits: launches one thread that waits on a shared-memory
 * mbarrier nothing ever arrives on.  After about one second the wait gives up,
 * sets the status word and the kernel returns normally (no trap, no fault; the
 * context stays usable).  The next dit_last_device_status() on the same
 * stream then returns DIT_ERR_DEVICE_TIMEOUT.  Diagnostic only; the pages
 * have no counterpart (they detect slow devices at the scheduling level).
 */
dit_status dit_selftest_bounded_wait(dit_stream_t stream);

/* Static English text for a status code; never NULL. */
const char *dit_status_string(dit_status status);

/* Version of this ABI (incremented on any signature change). */
int dit_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DIT_ATTN_H */
