/*
 * fa.h — C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * The operation: the fused, tiled, exact multi-head attention forward pass
 *
 *     O   = softmax(scale * Q K^T  [+ causal mask]) V
 *     LSE = per-row log-sum-exp of the scaled, masked scores (natural log)
 *
 * as computed by the forward kernel of "flash_attention_2.cu"
 * (leloykun/flash-hyperbolic-attention-minimal): scores are scaled before the
 * row max, the softmax runs online over key tiles (running max m and sum l,
 * partial O rescaled by exp(m_old - m_new)), and the kernel returns
 * O = O / l together with L = m + log(l).  The loop order is the swapped one
 * of "parallel execution of read/write operations (paper vs implementation)"
 * (query tile outer, key tiles inner, O written once), and the grid runs over
 * queries as well as batch and heads, as in "Meta's xFormers has Attention
 * kernel written in CUTLASS" (forward parallelised across the queries).
 * fa_bwd computes its gradients (dq, dk, dv) for an upstream gradient.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout:   q [B, H, Nq, d]; k, v [B, H, Nk, d]; o [B, H, Nq, d];
 *           lse [B, H, Nq]; all contiguous, row-major (d fastest).  The
 *           element (b, h, n, x) of q sits at ((b*H + h)*Nq + n)*d + x.
 * Types:    dtype FA_DTYPE_BF16      q, k, v, o are bf16; fp32 accumulation.
 *           dtype FA_DTYPE_F32       q, k, v, o are fp32; tensor-core TF32
 *                                    products, fp32 accumulation; the
 *                                    scores as three tf32 products of the
 *                                    split operands (hi/lo), P and V in tf32.
 *           dtype FA_DTYPE_F32_SIMT  q, k, v, o are fp32; plain fp32 FMA
 *                                    kernel, no tensor cores.
 *           dtype FA_DTYPE_F16       q, k, v, o are fp16; fp32 accumulation
 *                                    (the bf16 kernels with fp16 operands).
 *           lse is always fp32, natural log, in units of the scaled score.
 * Masking:  causal = 1 keeps key j for query i iff j <= i (top-left aligned,
 *           the rule of the forward kernel of "flash_attention_2.cu").  Keys
 *           j >= Nk never take part; rows i >= Nq are not written.
 * Scale:    any finite float; it multiplies q.k before the softmax.
 * Streams:  `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *           default stream.  Work is enqueued asynchronously on that stream.
 *           The forward kernels are launched with programmatic stream
 *           serialization: a CTA may start its set-up (shared and tensor
 *           memory, barriers) while the previous kernel on the stream is
 *           still running, but it reads and writes no global memory before
 *           that kernel has completed, so stream order holds for every
 *           buffer as with a plain launch.
 * Ownership: the caller owns every buffer.  The library never frees caller
 *           memory and never keeps a pointer after the call returns.  Its
 *           only allocation is one small per-device status buffer, made with
 *           cudaMalloc on the first call on each device and kept until exit.
 * Errors:   every function returns an fa_status code; nothing is printed and
 *           nothing aborts the process.
 * Threads:  entry points are reentrant; calls on different streams may run
 *           concurrently.  The status word is shared per device.
 */
#ifndef FA_H
#define FA_H

#ifdef __cplusplus
extern "C" {
#endif

#define FA_VERSION 10000 /* 1.0.0 */

/* The library is built with hidden symbol visibility (-fvisibility=hidden);
 * only the functions declared here are exported, so two builds loaded in one
 * process (the release and the debug library) share no internal symbols. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

typedef enum {
    FA_DTYPE_BF16 = 0,
    FA_DTYPE_F32 = 1,
    FA_DTYPE_F32_SIMT = 2,
    FA_DTYPE_F16 = 3
} fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, size < 1, bad flag,
                                  non-finite scale, overlapping buffers       */
    FA_ERR_UNSUPPORTED = 2,    /* valid problem outside the compiled set, e.g.
                                  head dim, or a device that is not sm_103    */
    FA_ERR_CUDA = 3,           /* a CUDA runtime call or a launch failed      */
    FA_ERR_DEVICE_TIMEOUT = 4  /* a kernel gave up waiting (see fa_fwd_status)*/
} fa_status;

/*
 * fa_fwd — attention forward on device buffers.
 *
 * q, k, v   device pointers to the inputs (layout above), 16-byte aligned.
 * o         device pointer to the output, 16-byte aligned; must not overlap
 *           q, k, v or lse.  It need not be zeroed: every element of every
 *           row i < Nq is written.
 * lse       device pointer to B*H*Nq floats, 4-byte aligned; every entry is
 *           written.
 * B, H      batch size and number of heads, 1 .. 65535 each, with
 *           B * H <= 2^31 - 1 (else FA_ERR_INVALID_ARG).
 * Nq, Nk    query and key sequence lengths, >= 1 (ragged lengths allowed).
 * d         head dimension.  FA_DTYPE_BF16, FA_DTYPE_F16: 32, 64, 128 or 256.
 *           FA_DTYPE_F32: 32, 64 or 128.
 *           FA_DTYPE_F32_SIMT: 1 .. 128.  Anything else is
 *           FA_ERR_UNSUPPORTED (the role of the "Failed to find groupsize ...
 *           Shared Memory constraint" error of "Flash Attention Shared Memory
 *           constraint", returned rather than raised).
 * scale     finite multiplier of q.k (commonly 1/sqrt(d)).
 * causal    0 or 1.
 * dtype     an fa_dtype value.
 * stream    cudaStream_t (as void*), or NULL.
 *
 * Returns FA_OK once the work is enqueued; argument errors are detected on
 * the host before anything is enqueued.  A kernel that stops waiting on one of
 * its internal barriers (a bounded wait, about two seconds) records it in the
 * per-device status word; read it with fa_fwd_status.
 */
FA_API int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int H, int Nq, int Nk, int d, float scale, int causal,
           int dtype, void *stream);

/*
 * fa_fwd_noalloc — fa_fwd for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for how the
 * library is deployed, not for the method.
 *
 * fa_fwd obtains its per-device status word with cudaMalloc on its first call
 * on each device.  Some callers cannot allow that: a serving process that
 * reserves all of the GPU's memory for its own pool at start-up, a
 * latency-critical loop that must not pay the device-wide synchronisation a
 * cudaMalloc implies, or a framework whose memory manager has to account for
 * every device allocation.  This entry point runs the same kernels but keeps
 * the status word in a fixed 256-byte array that is part of the library's
 * device image (every GPU that loads the library holds it until exit), and
 * calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments q .. stream are those of fa_fwd, with the same layout, alignment
 * and validation.  The scratch this call needs is one status word whatever the
 * problem size; a need beyond the 256-byte array would be refused with
 * FA_ERR_UNSUPPORTED before anything is enqueued.
 * device_status  NULL: the call returns once the work is enqueued and does
 *                not report the status word.  A bounded-wait give-up in this
 *                form reaches no one: the word stays in the array until the
 *                next call clears it (fa_fwd_status reads fa_fwd's word, not
 *                this one), so callers that need the report use the waiting
 *                form.  Non-NULL: the call waits for the
 *                stream, stores the raw status word there (bits as in
 *                fa_fwd_status) and returns FA_ERR_DEVICE_TIMEOUT if it is
 *                non-zero.
 * Set-up: the first call on each device looks up the array's device address
 * (with that device current); make that first call before any stream capture.
 * Sharing: every call uses the same array and clears the status word on its
 * stream before launching; calls whose work overlaps on the GPU (different
 * streams, or another thread) race on that word, so serialise them.
 */
FA_API int fa_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int H, int Nq, int Nk, int d, float scale, int causal,
                   int dtype, void *stream, int *device_status);

/*
 * fa_fwd_splitkv — fa_fwd with the key range of every query tile split into
 * chunks that run as separate CTAs, then merged.  For grids too small to fill
 * the GPU (few heads and few query tiles, e.g. short queries against long
 * keys): one CTA per (batch, head, query tile) leaves most SMs idle, which the
 * per-head parallelism of "parallel execution of read/write operations (paper
 * vs implementation)" already needs B*H of about 80 to avoid.  Each chunk
 * keeps its own running max and sum; the merge is the same online-softmax
 * update applied across chunks: LSE = log sum_s e^{LSE_s},
 * O = sum_s e^{LSE_s - LSE} O_s.
 *
 * Arguments q .. dtype and stream as for fa_fwd (tensor-core dtypes only;
 * FA_DTYPE_F32_SIMT is FA_ERR_UNSUPPORTED).
 * num_splits       chunks per query tile, 1 .. 64, or 0 to choose one wave of
 *                  about one CTA per SM (limited to what the workspace holds).
 *                  1 (or a choice of 1) runs fa_fwd itself.
 * workspace        caller-owned device memory, 256-byte aligned, of at least
 *                  fa_fwd_splitkv_workspace(B, H, Nq, d, num_splits) bytes;
 *                  it must not overlap q, k, v, o or lse.  It holds fp32
 *                  partial outputs between the two kernels of one call; calls
 *                  that share a workspace must not overlap on the GPU.
 * workspace_bytes  its size.
 * Returns FA_ERR_INVALID_ARG for a missing, misaligned or too small workspace
 * (when num_splits > 1), before anything is enqueued.
 */
FA_API int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int H, int Nq, int Nk, int d, float scale, int causal,
                   int dtype, int num_splits, void *workspace,
                   unsigned long long workspace_bytes, void *stream);

/* Bytes of workspace fa_fwd_splitkv needs for num_splits chunks (1 .. 64):
 * num_splits * B * H * Nq * (d + 1) floats, each part rounded up to 256
 * bytes.  0 for invalid arguments. */
FA_API unsigned long long fa_fwd_splitkv_workspace(int B, int H, int Nq, int d, int num_splits);

/*
 * fa_fwd_varlen — the forward over a batch of sequences of different lengths
 * packed end to end, each attending only within itself (the "variable
 * sequence length" case of "Meta's xFormers has Attention kernel written in
 * CUTLASS").  Causal masking is top-left within each sequence.
 *
 * Layout (token-major, heads interleaved):
 *   q, o [total_q, H, d]; k, v [total_k, H, d]; lse [H, total_q] (fp32).
 * cu_seqlens_q, cu_seqlens_k  device int32 arrays of B+1 offsets: sequence b
 *   holds rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) of q/o and
 *   [cu_seqlens_k[b], cu_seqlens_k[b+1]) of k/v; nondecreasing, starting at
 *   0 and ending at total_q / total_k.  They are read on the device, so they
 *   are not checked on the host; the kernels clamp every offset to
 *   [0, total_q] or [0, total_k], so whatever they hold no row past total_q
 *   or total_k is read or written and no sequence spans more rows than
 *   exist, but wrong offsets give wrong results.
 * max_seqlen_q  the longest query length (sizes the grid; 1 .. total_q).
 * A sequence with queries and no keys gets O = 0 and LSE = -inf.
 * Other arguments as for fa_fwd (tensor-core dtypes only; the SIMT dtype is
 * FA_ERR_UNSUPPORTED).  All pointers 16-byte aligned except lse and the
 * offsets (4 bytes).
 */
FA_API int fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                  const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int H,
                  int total_q, int total_k, int max_seqlen_q, int d, float scale,
                  int causal, int dtype, void *stream);

/*
 * fa_fwd_staged — the forward with a caller-provided staging area.  For
 * FA_DTYPE_F32 a pre-pass splits K into bf16 halves K_hi = bf16(K) and
 * K_lo = bf16(K - K_hi) and writes V, rounded to tf32 and transposed, into
 * the K-major V^T layout the tf32 P V product (tcgen05 kind::tf32) takes,
 * once per call; the kernel then loads them ready-made instead of every
 * query-tile CTA converting the same tiles again.  The kernel splits Q the
 * same way and computes the scores as three bf16 products (kind::f16),
 * Q_hi K_hi + Q_hi K_lo + Q_lo K_hi: about 2^-16 of each term left out,
 * against 2^-22 for fa_fwd's three tf32 products, at twice the tensor rate.
 * Results therefore differ slightly from fa_fwd's; both meet the fp32
 * tolerances (max |dO| 5e-3, |dLSE| 1e-3).  Other dtypes have nothing to
 * stage and run fa_fwd (workspace may then be NULL).
 *
 * Arguments q .. dtype and stream as for fa_fwd.
 * workspace        FA_DTYPE_F32: caller-owned device memory, 256-byte
 *                  aligned, of at least fa_fwd_staged_workspace(B, H, Nk, d,
 *                  dtype) bytes, not overlapping q, k, v, o or lse.  Calls
 *                  that share a workspace must not overlap on the GPU.
 * Returns FA_ERR_INVALID_ARG for a missing, misaligned, short or overlapping
 * workspace (fp32), before anything is enqueued.
 */
FA_API int fa_fwd_staged(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int H, int Nq, int Nk, int d, float scale, int causal,
                  int dtype, void *workspace, unsigned long long workspace_bytes,
                  void *stream);

/* Bytes of workspace fa_fwd_staged needs: for FA_DTYPE_F32, twice B*H*Nk*d
 * bf16 values (K_hi and K_lo) plus B*H*d*ceil(Nk/128)*128 floats (V^T), each
 * part rounded up to 256 bytes; 0 for other dtypes and for invalid
 * arguments. */
FA_API unsigned long long fa_fwd_staged_workspace(int B, int H, int Nk, int d, int dtype);

/*
 * fa_bwd — gradients of the forward for an upstream gradient dout: the
 * backward kernel of "flash_attention_2.cu"
 * (leloykun/flash-hyperbolic-attention-minimal), with the probabilities
 * recomputed from the saved log-sum-exp:
 *   P = exp(scale * Q K^T - LSE) (causal keys masked),  D = rowsum(dout * o),
 *   dv = P^T dout,  dS = P * (dout V^T - D),  dq = scale * dS K,
 *   dk = scale * dS^T Q.
 *
 * q, k, v, o, lse  the forward's inputs and outputs, as for fa_fwd (o and
 *                  lse must come from fa_fwd, or hold the same values).
 * dout             upstream gradient [B,H,Nq,d], the type of q.
 * dq [B,H,Nq,d], dk and dv [B,H,Nk,d]: outputs, the type of q, every element
 *                  written (keys that no query sees get zero gradients).
 * dtype            FA_DTYPE_BF16 or FA_DTYPE_F16 with d 32, 64 or 128 (tcgen05
 *                  kind::f16; P and dS are rounded to the input type, the
 *                  products accumulate in fp32), or FA_DTYPE_F32 /
 *                  FA_DTYPE_F32_SIMT with d 1 .. 128 (fp32 on the CUDA cores:
 *                  dq, dk, dv fp32, dq accumulated with atomic adds, so its
 *                  last bits may differ between runs); anything else is
 *                  FA_ERR_UNSUPPORTED.
 * workspace        caller-owned device memory, 256-byte aligned, of at least
 *                  fa_bwd_workspace(B, H, Nq, d) bytes: an fp32 dq
 *                  accumulator and two fp32 values per query row.  Calls that
 *                  share a workspace must not overlap on the GPU.
 * All pointers 16-byte aligned except lse (4 bytes); outputs and workspace
 * must not overlap each other or any input.  Asynchronous on `stream` (16-bit:
 * three kernels, per-row D and LSE, the tensor-core kernel, dq rounding;
 * fp32: two, per-row D with dq zeroed, the gradient kernel); bounded waits
 * report through the status word (fa_fwd_status).  Arguments are checked
 * before anything is enqueued (FA_ERR_INVALID_ARG).
 */
FA_API int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv,
           int B, int H, int Nq, int Nk, int d, float scale, int causal, int dtype,
           void *workspace, unsigned long long workspace_bytes, void *stream);

/* Bytes of workspace fa_bwd needs: B*H*Nq*max(d, 64) floats (the dq
 * accumulator, rows of the gradient kernel's head dim) plus
 * 2*B*H*ceil(Nq/128)*128 floats, each part rounded up to 256 bytes.  0 for
 * invalid arguments. */
FA_API unsigned long long fa_bwd_workspace(int B, int H, int Nq, int d);

/*
 * fa_bwd_varlen — fa_bwd over a batch of sequences of different lengths
 * packed end to end (the layout of fa_fwd_varlen): q, o, dout, dq
 * [total_q, H, d]; k, v, dk, dv [total_k, H, d]; lse [H, total_q] from
 * fa_fwd_varlen; cu_seqlens_q/k device int32 offsets (B+1 each, nondecreasing,
 * from 0 to total_q / total_k, covering every token: dq of rows outside
 * every sequence is unspecified).  Causal masking is top-left within each sequence;
 * keys that no query sees get zero dk, dv.  max_seqlen_q, max_seqlen_k: the
 * longest query and key lengths (1 .. total).  dtype, d, scale, causal as for
 * fa_bwd.  workspace: at least fa_bwd_varlen_workspace(B, H, total_q,
 * max_seqlen_q, d) bytes, 256-byte aligned (an fp32 dq accumulator and two
 * floats per padded query row).  The offsets are read on the device and not
 * checked on the host; every row index stays below total_q / total_k.
 */
FA_API int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse,
                  const void *dout, void *dq, void *dk, void *dv,
                  const int *cu_seqlens_q, const int *cu_seqlens_k, int B, int H,
                  int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                  float scale, int causal, int dtype, void *workspace,
                  unsigned long long workspace_bytes, void *stream);

/* Bytes of workspace fa_bwd_varlen needs: total_q*H*max(d, 64) floats plus
 * 2*H*B*ceil(max_seqlen_q/128)*128 floats, parts rounded up to 256 bytes;
 * 0 for invalid arguments. */
FA_API unsigned long long fa_bwd_varlen_workspace(int B, int H, int total_q, int max_seqlen_q, int d);

/*
 * fa_fwd_host — the same forward on HOST buffers.
 *
 * q_h, k_h, v_h   host inputs (pinned memory gives full copy speed).
 * o_h, lse_h      host outputs.
 * q_d .. lse_d    caller-owned device buffers of the same sizes, used as the
 *                 staging area; same alignment rules as fa_fwd.
 * The call splits the B*H planes into chunks (one per 64 MB of input, at
 * most eight) and pipelines them:
 * a chunk's inputs are copied host->device on an internal stream, its
 * forward runs on `stream` once they have landed, and its o, lse are copied
 * device->host on a second internal stream, so copies in, kernels and copies
 * out of different chunks overlap.  The internal streams and events are
 * created on first use per device and kept; concurrent calls on one device
 * are serialised.  Work already on `stream` completes before the inputs are
 * overwritten, and every enqueued step has finished when the call returns,
 * so the host outputs are ready on return.  Returns the first failing status.
 */
FA_API int fa_fwd_host(const void *q_h, const void *k_h, const void *v_h,
                void *o_h, float *lse_h,
                void *q_d, void *k_d, void *v_d, void *o_d, float *lse_d,
                int B, int H, int Nq, int Nk, int d, float scale, int causal,
                int dtype, void *stream);

/*
 * fa_fwd_status — synchronise `stream`, then read and clear the current
 * device's status word.  *device_status (may be NULL) receives the raw word:
 * 0 when every kernel finished normally; otherwise bit r set means a warp of
 * role r gave up on a bounded wait (1 = TMA producer, 2 = MMA issuer,
 * 4 = softmax/epilogue warps, 8 = fault injected by the test hook,
 * 16 = shared memory not aligned as the backward kernel needs, 32 = an index
 * check of the debug build failed and the access was skipped).
 * Returns FA_OK, FA_ERR_DEVICE_TIMEOUT (word != 0) or FA_ERR_CUDA.
 */
FA_API int fa_fwd_status(void *stream, int *device_status);

/* Human-readable name of an fa_status value (static storage). */
FA_API const char *fa_status_string(int status);

/* FA_VERSION of the compiled library. */
FA_API int fa_version(void);

/*
 * fa_set_test_hooks — testing aid, process-wide.
 * skip_v_load != 0 makes the next launches of the tensor-core kernels skip the
 * first V-tile load, so the MMA issuer's bounded wait runs out and the kernel
 * returns through its error path (status bit 8 plus the role bits).
 * wait_limit_ns sets the bounded-wait limit in nanoseconds (0 = default,
 * 2e9).  Returns FA_OK.
 */
FA_API int fa_set_test_hooks(int skip_v_load, unsigned long long wait_limit_ns);

/*
 * fa_debug_build — 1 for the debug build of the library (libfa_debug.so,
 * compiled with FA_DEBUG), 0 for the release build.  In the debug build the
 * kernels check the index of every plain global load and store they make
 * (the forward, the split-KV merge and the backward gradient kernel; TMA
 * copies are bounded by their tensor maps) against the buffer's extent: a
 * failed check skips the access and sets bit 32 in the status word that
 * fa_fwd_status reports.  No counterpart on the pages.
 */
FA_API int fa_debug_build(void);

/*
 * fa_set_debug_lse_shrink — testing aid of the debug build: the LSE extent
 * the index checks use is understated by `elems` entries (process-wide;
 * 0 restores it), so a test can see a check fire and the access skipped
 * without any access leaving a buffer.  Returns FA_OK, FA_ERR_INVALID_ARG
 * for elems < 0, or FA_ERR_UNSUPPORTED in the release build.
 */
FA_API int fa_set_debug_lse_shrink(long long elems);

/*
 * fa_set_fwd_schedule — testing aid, process-wide; no counterpart on the
 * pages (a scheduling choice of this implementation).  The bf16/fp16
 * forward of fa_fwd and fa_fwd_noalloc picks one of two schedules (see
 * fa_fwd_schedule).  block_items > 0 forces the blocked schedule with that
 * many items per CTA; otherwise ctas > 0 forces a persistent grid of that
 * many CTAs (at most one per item) and group_heads > 0 its planes per group
 * (at most all); zeros restore the automatic choice.  Results do not depend
 * on the schedule: every query tile does the same arithmetic wherever it
 * runs.  Returns FA_OK, or FA_ERR_INVALID_ARG for a negative argument.
 */
FA_API int fa_set_fwd_schedule(int ctas, int group_heads, int block_items);

/*
 * fa_fwd_schedule — the schedule fa_fwd would use for this problem on a GPU
 * with num_sms SMs; a host-only function, for reports and tests.  The
 * 16-bit forward runs a 1-D grid of *ctas CTAs over items (query tiles).
 *   *block_items = 0, persistent: about one CTA per SM; the planes are
 *     taken in groups of *group_heads whose K and V stay in L2 together
 *     (48 MB), within a group the items are dealt heaviest first, in rounds
 *     of *ctas items that go alternately to CTAs 0, 1, ... and ..., 1, 0.
 *   *block_items = G > 0, blocked: B*H*ceil(query tiles / G) CTAs, each
 *     taking G consecutive items of its plane's zigzag order (heaviest,
 *     lightest, ...), handed to SMs by the hardware as they free up.
 * The persistent schedule serves grids of up to 16 waves of items, the
 * blocked one larger grids.  *ctas = 0 for dtypes that run one CTA per
 * query tile.  Returns FA_OK, or FA_ERR_INVALID_ARG for null outputs, sizes
 * below 1 or causal not 0/1.
 */
FA_API int fa_fwd_schedule(int B, int H, int Nq, int Nk, int d, int causal, int dtype, int num_sms,
                    int *ctas, int *group_heads, int *block_items);

/*
 * fa_fwd_schedule_covers — host-only check of those schedules, for tests:
 * 1 if, for `planes` planes of n items on a grid of `ctas` CTAs (groups of
 * group_heads planes, block_items as above), every item is dealt to exactly
 * one CTA; else 0 (also for sizes below 1, a persistent grid with more CTAs
 * than items, a blocked grid of the wrong size, or more than 2^24 items).
 */
FA_API int fa_fwd_schedule_covers(int planes, int n, int ctas, int group_heads, int block_items);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
