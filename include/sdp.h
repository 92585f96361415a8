/*
 * sdp.h — C ABI of libsdp.so: fused grouped-query scaled-dot-product
 * attention forward for NVIDIA GB300 (sm_103a).
 *
 * The operation ("xe2-sdp-hd256" page, header and sections "HD=256
 * Architecture Differences" and "Performance Testing"; "xe2-sdp-bf16" page,
 * sections "Kernel Architecture: bf16io" and "Data flow diagram"): for batch
 * b, query head h, query row i, with G = Hq / Hkv and g = h / G,
 *
 *     s_j      = scale * <Q[b,h,i,:], K[b,g,j,:]>          0 <= j < Skv
 *     O[b,h,i] = sum_j softmax(s)_j * V[b,g,j,:]
 *     LSE      = ln sum_j exp(s_j)                         (natural log)
 *
 * The softmax statistics (row maximum, row sum) are kept in fp32; the two
 * contractions take fp16 or bf16 operands and accumulate in fp32. O has the
 * input dtype ("bf16io": bf16 in, bf16 out); LSE is fp32.
 *
 * Every pointer argument is plain memory; no framework type crosses this
 * boundary. The calls are not re-entrant on one stream in any special way:
 * each call only enqueues work on `stream`.
 */
#ifndef GQA_SDP_H
#define GQA_SDP_H

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes */
#define SDP_FP16 0
#define SDP_BF16 1

/* status codes (0 or negative) */
#define SDP_OK 0
#define SDP_ERR_INVALID_ARG (-1)    /* null pointer, non-positive size, Hq % Hkv != 0, non-finite scale, o aliasing q/k/v */
#define SDP_ERR_UNSUPPORTED (-2)    /* D not 128 or 256, unknown dtype, device not sm_103 */
#define SDP_ERR_ALIGNMENT (-3)      /* q, k, v, o not 16-byte aligned, or lse not 4-byte aligned */
#define SDP_ERR_OVERFLOW (-4)       /* index space does not fit the kernel's 32-bit tile and coordinate counters */
#define SDP_ERR_CUDA (-5)           /* a CUDA runtime/driver call failed; sdp_last_cuda_error() gives the code */
#define SDP_ERR_DEVICE_TIMEOUT (-6) /* a kernel gave up on a bounded wait and flagged its status word */
#define SDP_ERR_BAD_SEQLENS (-7)    /* sdp_fwd_varlen: a kernel found bad sequence offsets (status word) */

/*
 * sdp_fwd — O = softmax(Q K^T * scale) V and LSE, enqueued on `stream`.
 *
 * q    device, [B, Hq, Sq, D], contiguous row-major, dtype elements
 * k, v device, [B, Hkv, Skv, D], contiguous row-major, dtype elements
 * o    device, [B, Hq, Sq, D], contiguous row-major, dtype elements (written)
 * lse  device, [B, Hq, Sq] fp32 (written), or NULL to skip it
 * B, Hq, Hkv, Sq, Skv >= 1 with Hq % Hkv == 0; D in {128, 256}
 * scale  finite fp32 multiplier of the scores (1/sqrt(D) is the usual value)
 * dtype  SDP_FP16 or SDP_BF16 (the type of q, k, v and o)
 * stream a cudaStream_t (NULL = the legacy default stream)
 *
 * Ownership: all buffers belong to the caller and must stay valid until the
 * enqueued work has finished. q, k, v are only read; o and lse are only
 * written (never read first). o must not alias q, k or v (rejected when the
 * pointers are equal; other overlaps are undefined).
 *
 * Errors: on any validation error nothing is launched and the code is
 * returned. SDP_ERR_CUDA reports a failed tensor-map encode or launch. The
 * call does not synchronise, so a device-side timeout is reported later by
 * sdp_poll_status(). On the first call on a device the library allocates its
 * status region there: the status word and 1024 unit-claim counters, 4100
 * bytes (freed by sdp_shutdown()); the allocation and its zeroing are
 * synchronous, so make that first call outside stream capture.
 *
 * Streams and graphs: calls on different streams, from any host threads, may
 * run at once. A host thread's first call may be its first CUDA work: the call
 * binds the current device's primary context to the thread (cudaSetDevice),
 * as the runtime itself does on a thread's first call that needs a context. Launches without the causal mask that run on single CTAs (head
 * dim 128, or a group size whose units do not pair) with more 128-row units
 * than SMs use a persistent kernel whose CTAs claim units from a counter of the
 * launching stream (streams get counters in the order they are first used,
 * found by the stream's unique id, cudaStreamGetId). A launch captured into a
 * CUDA graph, or on a stream after the 1024th, runs one CTA per unit instead:
 * the same results, bit for bit.
 */
int sdp_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
            int B, int Hq, int Hkv, int Sq, int Skv, int D, float scale, int dtype,
            void *stream);

/*
 * sdp_fwd_causal — sdp_fwd with causal masking: query row i attends to keys
 * 0..i only (top-left alignment, as PyTorch's is_causal; rows i >= Skv see
 * every key). The "SyclKittens" summary reports causal attention (sections
 * E.4, E.6) without fixing a convention. Same arguments, layout, ownership
 * and errors as sdp_fwd. Key tiles past a query tile's last row are skipped,
 * so the work is about half of sdp_fwd's when Sq = Skv.
 */
int sdp_fwd_causal(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int Hq, int Hkv, int Sq, int Skv, int D, float scale, int dtype,
                   void *stream);

/*
 * sdp_merge — combine partial results over disjoint key sets into the result
 * over their union: the state exchange of ring / context-parallel attention
 * ("SyclKittens" summary, section I.2). For every row r:
 *
 *     LSE[r] = ln sum_p exp(LSE_p[r]),    O[r,:] = sum_p exp(LSE_p[r] - LSE[r]) * O_p[r,:]
 *
 * o_parts   device, [nparts, rows, D] contiguous, dtype elements: each part's
 *           normalised output (e.g. sdp_fwd's o over one key shard)
 * lse_parts device, [nparts, rows] fp32: each part's log-sum-exp (sdp_fwd's
 *           lse); -inf marks a part without keys; at least one part per row
 *           must be finite
 * o         device, [rows, D] dtype (written); lse [rows] fp32 (written) or NULL
 * rows = B*H*Sq for sdp_fwd's layouts; D in {128, 256}; dtype SDP_FP16/BF16.
 * Weights and sums in fp32, output rounded to nearest even. Buffers 16-byte
 * aligned (lse 4-byte); o must not alias o_parts. Enqueued on `stream`;
 * validation errors launch nothing; a failed launch returns SDP_ERR_CUDA.
 */
int sdp_merge(const void *o_parts, const float *lse_parts, int nparts, long long rows, int D, int dtype,
              void *o, float *lse, void *stream);

/*
 * Split-KV forward, for problems with too few (batch, head, 128-row query
 * tile) units to occupy the GPU: decode (Sq = 1 or a few rows) and short
 * batches over long contexts. The "SyclKittens" summary's attention section
 * (E.4) adds a split-K variant and its dispatch section (E.5) picks the
 * kernel by query length and batch; here the keys are cut into n_splits
 * contiguous runs of 128-key tiles, each (unit, run) pair becomes one CTA
 * writing a partial O and LSE into the caller's workspace, and sdp_merge
 * combines the runs into o / lse. The result is the same function as
 * sdp_fwd's; the partial O is rounded to the I/O dtype once before the merge.
 *
 * sdp_fwd and sdp_fwd_splitkv both pack the G query heads of a KV group into
 * one head of G * Sq rows when Sq is not a multiple of 128 (no causal mask):
 * the same memory, viewed as [B, Hkv, G*Sq, D], so decode fills the tiles.
 *
 * sdp_fwd_splitkv_count — the split count a call with these sizes and
 * n_splits uses on the current device: n_splits = 0 picks the most that
 * still run in one wave of one CTA per SM; any request is clamped to
 * [1, ceil(Skv / 128)] and evened out. Returns the count (>= 1) or a negative status code.
 *
 * sdp_fwd_splitkv_workspace_bytes — the workspace such a call needs (0 when
 * the count is 1), or a negative status code.
 *
 * sdp_fwd_splitkv — sdp_fwd's arguments (no causal mask), plus
 *   n_splits        0 (automatic) or the requested count
 *   workspace       device scratch of at least the size above, 16-byte
 *                   aligned, owned by the caller, not overlapping q/k/v/o;
 *                   NULL allowed when the size is 0. Its contents on entry
 *                   do not matter; on exit they are unspecified.
 *   workspace_bytes its size
 * Errors as sdp_fwd, plus SDP_ERR_INVALID_ARG for a negative n_splits or a
 * missing / short / overlapping workspace. Two kernels are enqueued on
 * `stream` (attention, then sdp_merge); the library allocates nothing but
 * sdp_fwd's status word.
 */
int sdp_fwd_splitkv_count(int B, int Hq, int Hkv, int Sq, int Skv, int D, int dtype, int n_splits);
long long sdp_fwd_splitkv_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int D, int dtype, int n_splits);
int sdp_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                    int B, int Hq, int Hkv, int Sq, int Skv, int D, float scale, int dtype,
                    int n_splits, void *workspace, unsigned long long workspace_bytes, void *stream);

/*
 * sdp_fwd_varlen — attention over a batch of sequences of different lengths
 * packed back to back (no counterpart on the pages: the plain generalisation
 * of a ragged last tile to a batch of ragged sequences). Sequence b owns
 * query rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key rows
 * [cu_seqlens_k[b], cu_seqlens_k[b+1]); each query row attends to its own
 * sequence's keys only, as in sdp_fwd (causal != 0: row i of a sequence sees
 * that sequence's keys 0..i, top-left). A row of a sequence with no keys gets
 * O = 0 and LSE = -inf.
 *
 * q       device, [total_q, Hq, D] (token, head, dim), contiguous, dtype
 * k, v    device, [total_k, Hkv, D], contiguous, dtype
 * o       device, [total_q, Hq, D] (written); lse [Hq, total_q] fp32 or NULL
 * cu_seqlens_q, cu_seqlens_k  device int32 [nseq + 1]: 0, then non-decreasing
 *         offsets, ending at total_q / total_k
 * max_seqlen_q  host int >= every query length. Up to 512 sequences (64 with
 *         causal != 0) the grid holds only the 128-row tiles that exist, at
 *         most (total_q + 127 * nseq) / 128 per head, and each CTA finds its
 *         tile from the offsets; beyond that it holds the longest sequence's
 *         tiles for every (sequence, head)
 * Hq % Hkv == 0, D in {128, 256}; total_q == 0 returns SDP_OK at once (null
 * pointers allowed then), before the other checks.
 *
 * Ownership and aliasing as sdp_fwd. The offsets live on the device, so they
 * are checked by the kernel: a sequence whose offsets leave [0, total], go
 * down, or give more rows than max_seqlen_q rounded up to a multiple of 128
 * is not computed (nor, where offsets that go down make sequences overlap,
 * those past the grid's tile count), and the next sdp_poll_status returns
 * SDP_ERR_BAD_SEQLENS. Inputs must be finite: the key rows after a
 * sequence's last key in its last 128-key tile belong to the next sequence
 * and are read, with weight exactly 0. With an even number of query heads per
 * KV head, tiles run on CTA pairs (two heads of a group on one tile); tiles
 * that end past their sequence store O row by row.
 */
int sdp_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                   const int *cu_seqlens_q, const int *cu_seqlens_k, int nseq, int Hq, int Hkv,
                   int total_q, int total_k, int max_seqlen_q, int D, float scale, int dtype, int causal,
                   void *stream);

/*
 * sdp_fwd_noalloc — sdp_fwd for callers that cannot allocate device memory.
 * No page describes a counterpart: this is a library-usage variant, not a step of
 * the method.
 *
 * sdp_fwd allocates its 4100-byte status region on a device the first time it runs
 * there (cudaMalloc). Callers that cannot allow that use this entry point
 * instead: code running inside a memory pool or arena that owns all device
 * memory of the process, plugins whose host forbids allocations outside its
 * own allocator, and code paths where an allocation's implicit
 * synchronisation is not acceptable. This call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Arguments, layout, ownership, validation and results are those of sdp_fwd,
 * and the launch is sdp_fwd's own: the same head packing, the same kernel
 * choice, the same wait limit (sdp_set_wait_timeout_ms) and debug flags, so the
 * outputs are bit for bit those of sdp_fwd. The kernels' only scratch, the
 * status word and the unit-claim counters of the persistent single-CTA kernel
 * (1024 words, one per stream as for sdp_fwd, zeroed in stream order by the
 * launches that use them), lives in a static device array of
 * SDP_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads the
 * library holds until the process exits; sdp_fwd keeps the same region in its
 * per-device allocation. A launch needs 4 bytes of it for the status word
 * whatever the problem size.
 *
 * Set-up: the first call on each device (made with that device current)
 * looks up the device address of the array with cudaGetSymbolAddress and
 * caches it (sdp_shutdown forgets it); make that first call before any stream
 * capture.
 *
 * Sharing: every call in the process uses the same array. Each call clears
 * the status word on `stream` before its kernel (a 4-byte cudaMemsetAsync), so
 * calls that overlap on the GPU (different streams without ordering between
 * them) race on it. A wait that times out inside the kernel leaves its output
 * tile unwritten and records the event in that word, not in the word that
 * sdp_poll_status reads: read it with sdp_fwd_noalloc_status.
 */
#define SDP_NOALLOC_SCRATCH_BYTES 4352
int sdp_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                    int B, int Hq, int Hkv, int Sq, int Skv, int D, float scale, int dtype,
                    void *stream);

/*
 * sdp_fwd_noalloc_status — synchronise `stream`, then read and clear the status
 * word of sdp_fwd_noalloc's shared array on the current device (as the last
 * such call that finished left it). Allocates nothing (cudaMemcpyFromSymbol /
 * cudaMemcpyToSymbol of 4 bytes). Returns SDP_OK, SDP_ERR_DEVICE_TIMEOUT (a
 * wait gave up; the detail is then in sdp_last_status_detail) or SDP_ERR_CUDA.
 */
int sdp_fwd_noalloc_status(void *stream);

/*
 * sdp_poll_status — synchronise `stream`, then read and clear the current
 * device's status word. Returns SDP_OK, SDP_ERR_DEVICE_TIMEOUT (a kernel
 * abandoned a wait after the timeout and returned without writing its
 * tile), SDP_ERR_BAD_SEQLENS (sdp_fwd_varlen found bad offsets), or
 * SDP_ERR_CUDA (the synchronisation itself failed).
 */
int sdp_poll_status(void *stream);

/*
 * sdp_last_status_detail — the raw status word read by the last
 * sdp_poll_status() that found an error: bits 0-7 name the wait that timed
 * out (1 Q load, 2 KV slot empty, 3 KV slot full, 4 S ready, 5 P ready,
 * 6 O done) or 7 for bad sequence offsets, bits 8-31 the CTA index (saturating).
 */
unsigned int sdp_last_status_detail(void);

/*
 * sdp_set_wait_timeout_ms — upper bound, in milliseconds, on any single wait
 * inside the kernel (default 2000). Applies to launches made after the call.
 * Returns the previous value. 0 restores the default.
 */
unsigned int sdp_set_wait_timeout_ms(unsigned int ms);

/*
 * sdp_set_debug_flags — test hooks, 0 by default. Bit 0: the load warp issues
 * no copies at all, so every consumer wait runs out and the kernel returns
 * through its timeout path (used to test that path without a fault). Bit 1:
 * always run the single-CTA kernel, never the CTA-pair kernel (both compute
 * the same result; tests compare them). Bit 2: never pack the query heads of
 * a group into one head (same result; tests compare). Bit 3: at head dim 128,
 * use the CTA-pair kernel where it qualifies (by default head dim 128 runs on
 * single CTAs, which measured as fast or faster there). Bit 4: one CTA (or CTA
 * pair) per unit even where a persistent kernel applies (same result, bit for
 * bit). Bit 5: variable-length launches cover the longest sequence's query
 * tiles for every sequence instead of the list of tiles that exist (same
 * result, bit for bit). Bit 6: at head dim 128, never the two-tile CTA-pair
 * kernel. Bit 7: at head dim 128, run dense non-causal launches whose two-tile
 * units pair up on the two-tile CTA-pair kernel (two 128-row query tiles per
 * CTA, 64-key softmax steps; the same function, rounded differently), even
 * below one wave of CTAs. Returns the previous flags.
 */
int sdp_set_debug_flags(int flags);

/* The CUDA error code (cudaError_t) of the last SDP_ERR_CUDA in this process. */
int sdp_last_cuda_error(void);

/* A static, human-readable description of a status code. */
const char *sdp_strerror(int code);

/* ABI version: 100 * major + minor (101: sdp_fwd_causal; 102: sdp_merge; 103: split-KV; 104: varlen;
 * 105: sdp_fwd_noalloc_status; 106: SDP_NOALLOC_SCRATCH_BYTES 4352, the status region holds the
 * persistent single-CTA kernel's claim counters; 107: one claim counter per stream, captured
 * launches on the per-unit grid). */
int sdp_version(void);

/* Free the per-device status words and forget the cached tensor maps (host
 * copies of TMA descriptors, keyed by buffer address and shape). Call only with
 * no sdp work in flight. */
void sdp_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_SDP_H */
