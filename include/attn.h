/*
 * attn.h - C ABI of libattn.so: exact scaled-dot-product attention on GB300 (sm_103a).
 *
 * Forward:  O = softmax(scale * Q K^T [causal mask]) V, plus the per-row logsumexp L.
 * Backward: dQ, dK, dV of sum(dO * O), recomputing the probabilities from L.
 *
 * The operations are the ones described on these pages:
 *   - "Triton 05: Flash Attention" (wonbeomjang.kr): sections Online Softmax,
 *     코드 라인별 설명 (Forward), Backward 구현 (LSE로 P 재계산, Softmax Gradient,
 *     3단계 커널 구조) and torch.autograd.Function 래핑, which fixes the interface
 *     forward(q, k, v, causal) -> o (saving q, k, v, o, lse) and
 *     backward(do) -> dq, dk, dv with sm_scale = d ** -0.5.
 *   - "FlashAttentionを1から — 計算を増やして速くする逆説": sections オンラインsoftmax
 *     and 逆伝播で、わざと計算し直す (recompute P in the backward instead of storing it).
 *
 * Conventions shared by every entry point
 *   Layout   q, k, v, o, dO, dq, dk, dv are contiguous [B, H, N, d] tensors of 16-bit
 *            floats (fp16 or bf16, one type for all of them), row-major, d innermost.
 *            lse and the backward workspace are contiguous [B, H, N] float32.
 *            Every pointer is a DEVICE pointer, 16-byte aligned.
 *   Sizes    B >= 1, H >= 1, 1 <= N <= 1048576, B*H <= 65535; d a multiple of 8 from 8
 *            to 256 (split-KV decoding: d in {64, 128, 256}). The kernels are 64, 128 or 256
 *            columns wide: a smaller d runs on the next width with the missing columns
 *            read as zero (exact: they add zeros to every product) and never written, so
 *            d = 96 costs what d = 128 costs. The 256-column kernels take 128 query rows
 *            and 64-key blocks per step and run the dK/dV stage as two passes (dV, then
 *            dK), since the two accumulators do not fit in tensor memory together.
 *   Mask     causal != 0 masks key j for query i when j > i (top-left aligned,
 *            N_q = N_k, diagonal kept), so no row is ever fully masked.
 *   scale    the factor applied to Q K^T; finite and > 0 (the usual value is
 *            1/sqrt(d)).
 *   Streams  cuda_stream is a cudaStream_t (NULL = legacy default stream). All work
 *            is enqueued on it; the calls never synchronise the device and return
 *            as soon as the launches are queued.
 *   Ownership the caller allocates and owns every buffer and the stream. The library
 *            allocates no device memory and keeps no per-call state (tensor maps
 *            are encoded per call). Its device globals, one copy per device and
 *            shared by every call in the process, are the status words described
 *            under Errors and the 16 MiB array g_bwd_scratch that attn_bwd_noalloc
 *            keeps its D values in. Its host-side caches (the last schedule table
 *            of each persistent kernel, attn_step_host's side streams and events,
 *            attn_bwd_noalloc's array addresses) are guarded by locks. The calls
 *            may be made from several host threads; but calls whose work can
 *            overlap on the GPU share the status words, so attn_last_kernel_status
 *            then reports the first timeout of any of them, and they race on
 *            g_bwd_scratch if both are attn_bwd_noalloc.
 *   Errors   ATTN_ERR_INVALID_ARG for a bad size, pointer, alignment, scale or an
 *            output that overlaps an input (checked on the host before any CUDA
 *            call); ATTN_ERR_UNSUPPORTED for a head dimension or type the kernels do
 *            not implement; ATTN_ERR_CUDA when a launch or a tensor-map encoding
 *            fails (the CUDA error is then also left for cudaGetLastError).
 *            Faults inside a kernel surface, as with any CUDA library, at the
 *            caller's next synchronisation. Every pipeline wait inside the kernels
 *            is bounded; a wait that runs out records ATTN_ERR_TIMEOUT in the
 *            status word read by attn_last_kernel_status().
 *   Environment (read once per process; every setting gives the same bits)
 *            ATTN_WAIT_LIMIT_CYCLES  SM cycles one pipeline wait may take (default
 *                                    2^31, about a second).
 *            ATTN_FWD_PERSISTENT, ATTN_BWD_PERSISTENT = 0 / 1  force the one-CTA-per-item
 *                                    or the persistent kernels (default: by shape).
 *            ATTN_FWD_PAIR = 1       run the 128-column forward on CTA pairs (two SMs
 *                                    sharing each K/V block through tcgen05 MMAs with
 *                                    cta_group::2); off by default, since on the
 *                                    measured shapes it is slower.
 *            For failure tests only: ATTN_TEST_STALL = 1 makes every kernel withhold
 *            its copies, so that its waits run out after ATTN_WAIT_LIMIT_CYCLES and
 *            every call reports ATTN_ERR_TIMEOUT (no results are computed).
 */
#ifndef ATTN_H
#define ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,
  ATTN_ERR_UNSUPPORTED = 2,
  ATTN_ERR_CUDA = 3,
  ATTN_ERR_TIMEOUT = 4
} attn_status;

typedef enum { ATTN_FP16 = 0, ATTN_BF16 = 1 } attn_dtype;

/*
 * attn_fwd - forward pass.
 * Computes, for every (b, h) slice and query row i,
 *   S_ij = scale * q_i . k_j  (S_ij = -inf for j > i when causal),
 *   O_i  = sum_j softmax(S_i)_j v_j,   L_i = max_j S_ij + ln sum_j exp(S_ij - max_j S_ij),
 * tile by tile with the online-softmax recurrence (running max m, denominator l,
 * unnormalised accumulator rescaled by exp(m_old - m_new), one final divide by l), so
 * that the N x N scores never reach device memory ("Triton 05: Flash Attention",
 * sections Online Softmax and 코드 라인별 설명 (Forward); "FlashAttention·FA4·FP4",
 * section 온라인 softmax가 블록 사이의 값을 어떻게 이어 주나).
 *   q, k, v  in:  [B, H, N, d] 16-bit.
 *   o        out: [B, H, N, d] same type as q.
 *   lse      out: [B, H, N] float32, natural-log L_i (the value attn_bwd consumes).
 * o and lse must not overlap q, k, v or each other.
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int N, int d, attn_dtype dtype, int causal,
                     float scale, void* cuda_stream);

/*
 * attn_bwd_workspace_bytes - bytes of the float32 workspace attn_bwd needs:
 * 4 * B * H * N (one D_i per query row). Returns 0 for non-positive sizes.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int N);

/*
 * attn_bwd - backward pass, three kernels on cuda_stream with no atomics
 * ("Triton 05: Flash Attention", section 3단계 커널 구조):
 *   1. D_i = rowsum(dO_i * O_i) into the workspace (section Softmax Gradient);
 *   2. per block of keys j: P_ij = exp(S_ij - L_i), dV_j = sum_i P_ij dO_i,
 *      dS_ij = P_ij (dO_i . v_j - D_i), dK_j = scale * sum_i dS_ij q_i;
 *   3. per block of queries i: dQ_i = scale * sum_j dS_ij k_j.
 *   q, k, v, o, dO in: [B, H, N, d] 16-bit; lse in: [B, H, N] float32 from attn_fwd
 *                      with the same q, k, v, causal and scale.
 *   dq, dk, dv    out: [B, H, N, d] same type as q.
 *   workspace     scratch of attn_bwd_workspace_bytes(B, H, N) bytes, device memory
 *                 owned by the caller; its contents on entry do not matter.
 * Outputs must not overlap the inputs, each other or the workspace.
 */
attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dO, void* dq, void* dk, void* dv,
                     void* workspace, int B, int H, int N, int d, attn_dtype dtype,
                     int causal, float scale, void* cuda_stream);

/*
 * attn_fwd_qk / attn_bwd_qk - attn_fwd and attn_bwd for N_q query rows against N_k keys
 * (a query chunk attending to a longer key sequence, as in chunked prefill):
 *   q, o, dO, dq  [B, H, Nq, d];  k, v, dk, dv  [B, H, Nk, d];  lse, workspace [B, H, Nq]
 * Causal masking is bottom-right aligned: the queries are the last Nq positions of the
 * sequence, key j is visible to query i iff j <= i + (Nk - Nq) (the pages' "future tokens
 * are blocked", "Triton 05: Flash Attention", section Causal Masking, read for a query
 * chunk that follows the keys already in the cache); causal requires Nk >= Nq
 * (ATTN_ERR_INVALID_ARG otherwise), so no row is fully masked. With Nq = Nk these are
 * exactly attn_fwd and attn_bwd. Everything else as for attn_fwd / attn_bwd.
 */
attn_status attn_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int H, int Nq, int Nk, int d, attn_dtype dtype, int causal,
                        float scale, void* cuda_stream);
attn_status attn_bwd_qk(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* dO, void* dq, void* dk, void* dv,
                        void* workspace, int B, int H, int Nq, int Nk, int d,
                        attn_dtype dtype, int causal, float scale, void* cuda_stream);

/*
 * attn_fwd_varlen / attn_bwd_varlen - attn_fwd and attn_bwd over a batch of sequences of
 * different lengths packed along the token axis, with no padding ("FlashAttentionを1から
 * — 計算を増やして速くする逆説", section 現場ではこう使う: padding sentences to the
 * longest one pays for the padded positions; the variable-length interface takes the
 * boundaries as cu_seqlens instead).
 *   q, o, dO, dq        [total_q, H, d] 16-bit, token-major (d innermost);
 *   k, v, dk, dv        [total_k, H, d];
 *   lse, workspace      [H, total_q] float32 (attn_bwd_varlen_workspace_bytes);
 *   cu_seqlens_q/_k     int32 [B + 1] in DEVICE memory, 4-byte aligned: sequence b owns
 *                       query tokens cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key tokens
 *                       cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1;
 *   cu_seqlens_q_host/_k_host  optional (both NULL, or both set) HOST copies of the same
 *                       B + 1 offsets, read during the call. They only order the work: the
 *                       persistent kernels then walk their items longest first, balanced
 *                       over the SMs, instead of in a fixed order (the sequences' lengths
 *                       differ, so a fixed order leaves some SMs working long after the
 *                       rest). Results do not depend on them: every item is computed,
 *                       whatever they say, from the device copies.
 *   max_seqlen_q/_k     bounds on every sequence's query / key count (1 .. 1048576, at
 *                       most the totals); the grids cover this many rows per sequence.
 * Each (sequence, head) pair is its own attention problem; causal masking is bottom-right
 * aligned within the sequence, as for attn_fwd_qk. Tokens outside every sequence are
 * neither read as queries nor written. A sequence with keys and no queries gets zero dk,
 * dv. The sizes are checked on the host (ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED as
 * for attn_fwd). cu_seqlens are read on the device, without synchronising: a sequence
 * that leaves its tensor, exceeds max_seqlen, has queries but no key, or (causal) fewer
 * keys than queries is skipped (its outputs are not written) and attn_last_kernel_status
 * then returns ATTN_ERR_INVALID_ARG.
 */
size_t attn_bwd_varlen_workspace_bytes(int H, int total_q); /* 4 * H * total_q; 0 if invalid */
attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens_q, const int* cu_seqlens_k,
                            const int* cu_seqlens_q_host, const int* cu_seqlens_k_host, int B,
                            int H, int total_q, int total_k, int max_seqlen_q,
                            int max_seqlen_k, int d, attn_dtype dtype, int causal, float scale,
                            void* cuda_stream);
attn_status attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dO, void* dq, void* dk, void* dv,
                            void* workspace, const int* cu_seqlens_q, const int* cu_seqlens_k,
                            const int* cu_seqlens_q_host, const int* cu_seqlens_k_host, int B,
                            int H, int total_q, int total_k, int max_seqlen_q,
                            int max_seqlen_k, int d, attn_dtype dtype, int causal, float scale,
                            void* cuda_stream);

/*
 * attn_bwd_preprocess - step 1 of attn_bwd alone: delta[b,h,i] = sum_c dO[b,h,i,c] *
 * o[b,h,i,c] in float32 ("Triton 05: Flash Attention", section 3단계 커널 구조,
 * [1단계] Preprocess). o, dO: [B, H, N, d] 16-bit device; delta: [B, H, N] float32
 * device, must not overlap o or dO.
 */
attn_status attn_bwd_preprocess(const void* o, const void* dO, float* delta, int B, int H,
                                int N, int d, attn_dtype dtype, void* cuda_stream);

/*
 * attn_bwd_dkv - step 2 of attn_bwd alone ("Triton 05: Flash Attention", section
 * 3단계 커널 구조, [2단계] dKV 커널): one CTA per block of 128 keys of one (b, h) slice
 * holds K_j, V_j on chip and loops over the query blocks that see them:
 *   P_ij = exp(S_ij - L_i), dV_j = sum_i P_ij dO_i, dS_ij = P_ij (dO_i . v_j - D_i),
 *   dK_j = scale * sum_i dS_ij q_i.
 * q, k, v, dO: [B, H, N, d] 16-bit; lse, delta: [B, H, N] float32 (delta from
 * attn_bwd_preprocess); dk, dv: [B, H, N, d] outputs, must not overlap any input or
 * each other. All device pointers, 16-byte aligned.
 */
attn_status attn_bwd_dkv(const void* q, const void* k, const void* v, const float* lse,
                         const float* delta, const void* dO, void* dk, void* dv, int B, int H,
                         int N, int d, attn_dtype dtype, int causal, float scale,
                         void* cuda_stream);

/*
 * attn_bwd_dq - step 3 of attn_bwd alone ("Triton 05: Flash Attention", section
 * 3단계 커널 구조, [3단계] dQ 커널): one CTA per block of 128 query rows holds Q_i and
 * dO_i on chip and loops over the visible key blocks: dQ_i = scale * sum_j dS_ij k_j.
 * Same inputs as attn_bwd_dkv; dq: [B, H, N, d] output that must not overlap them.
 */
attn_status attn_bwd_dq(const void* q, const void* k, const void* v, const float* lse,
                        const float* delta, const void* dO, void* dq, int B, int H, int N,
                        int d, attn_dtype dtype, int causal, float scale, void* cuda_stream);

/*
 * attn_bwd_noalloc - attn_bwd for callers that cannot allocate device memory, such as a
 * plugin inside a host engine that owns all device memory and offers no allocator or
 * workspace, or a serving loop that forbids cudaMalloc after start-up because it can
 * synchronise the device and stall other streams. The pages have no counterpart: this
 * entry point exists only for such callers.
 * Same arguments, layouts, results and errors as attn_bwd, minus `workspace`: the D
 * values live in a float32 array of ATTN_NOALLOC_MAX_ROWS entries (16 MiB) inside the
 * library, in device memory that every GPU which loads the library reserves until the
 * process exits. B * H * N above ATTN_NOALLOC_MAX_ROWS returns ATTN_ERR_INVALID_ARG.
 * Neither the library nor this call allocates anything.
 * The first call in a CUDA context (the device's primary context, or one a host engine
 * created and made current) looks up the array's address in that context (a
 * cudaGetSymbolAddress, with that context current) and remembers it for later calls in
 * the same context; make that first call before any stream capture there. Every call shares the one array and it keeps the last call's
 * values: calls whose work can overlap on the GPU (other streams, or host threads with
 * no ordering between them) race on it and produce wrong gradients, so serialise them.
 * Nothing in it has to start at zero: each call writes every entry it reads.
 */
#define ATTN_NOALLOC_MAX_ROWS 4194304
attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dO, void* dq, void* dk, void* dv,
                             int B, int H, int N, int d, attn_dtype dtype, int causal,
                             float scale, void* cuda_stream);

/*
 * attn_step_host - one training step of attention (attn_fwd then attn_bwd) on data that
 * lives in HOST memory: copies q, k, v, dO in, computes, and copies o, lse, dq, dk, dv out,
 * overlapping the copies with the kernels. The B*H slices are cut into `chunks` runs of
 * consecutive slices whose sizes ramp up and down (weights 1, 2, 3, 3, ..., 3, 2, 1): the
 * first upload and the last chunk's compute and download overlap nothing, so those chunks
 * are short. While chunk c is computed on cuda_stream, the inputs of chunk c + 1 are
 * copied in and the outputs of chunk c - 1 copied out on two side streams. Within a chunk
 * the forward waits only for Q, K and V (dO follows), and each output leaves as soon as
 * its kernel is done: O and L after the forward, dK and dV after their kernel, dQ last. The side
 * streams and the call's events are made on the first call in a CUDA context and kept for
 * later calls there until the process exits; a lock orders the enqueueing of concurrent
 * calls, whose copies then share the side streams. Results are identical to attn_fwd +
 * attn_bwd on
 * the whole tensors (every (b, h) slice is computed independently).
 *   q, k, v, dO        HOST [B, H, N, d] 16-bit inputs; pinned (page-locked) memory is
 *                      needed for the copies to overlap (pageable memory works, serially)
 *   o, dq, dk, dv, lse HOST outputs, [B, H, N, d] 16-bit and [B, H, N] float32
 *   scratch            DEVICE buffer of scratch_bytes >=
 *                      attn_step_host_scratch_bytes(B, H, N, d, chunks): two sets of
 *                      per-chunk device tensors (of the largest chunk), used in turn
 *   chunks             >= 1 (values above B*H are clamped)
 * Sizes, dtypes, scale and errors as for attn_fwd; every pointer 16-byte aligned. The
 * call only enqueues work: the outputs are valid once cuda_stream has completed it.
 */
size_t attn_step_host_scratch_bytes(int B, int H, int N, int d, int chunks); /* 0: invalid */
attn_status attn_step_host(const void* q, const void* k, const void* v, const void* dO,
                           void* o, float* lse, void* dq, void* dk, void* dv, void* scratch,
                           size_t scratch_bytes, int B, int H, int N, int d, attn_dtype dtype,
                           int causal, float scale, int chunks, void* cuda_stream);

/*
 * Split-KV decoding: one query row per (b, h) attending to all Nk keys of a K/V cache
 * (no mask), the keys split into ranges whose partial results are computed in parallel
 * and then joined. "FlashAttentionを1から — 計算を増やして速くする逆説", section
 * その後の版と、推論での事情: with a single query token the K/V side is split and the
 * partial results are combined with the online-softmax update equations (same page,
 * section オンラインsoftmax: 途中経過を、後から縮める), which gives the same answer as no
 * split.
 *
 *   q        [B, H, 1, d] 16-bit (fp16 or bf16, like k and v)
 *   k, v     [B, H, Nk, d] 16-bit, 1 <= Nk <= 1048576
 *   o        [B, H, 1, d] 16-bit: softmax(scale q K^T) V
 *   lse      [B, H] float32: L = m + ln l (natural log of the scaled scores)
 *   partials [B, H, num_splits, d + 4] float32 scratch owned by the caller
 *            (attn_decode_workspace_bytes); record s of a slice holds O~_s (d values,
 *            the unnormalised weighted sum of the split's value rows), m_s (its largest
 *            scaled score, natural-log units; -inf for an empty split), l_s (the sum of
 *            exp(scale s_j - m_s)) and two unused floats.
 *   num_splits 1 .. 65535. Split s covers keys [s C, min((s + 1) C, Nk)) with
 *            C = 64 * ceil(ceil(Nk / num_splits) / 64); splits past the end are empty.
 * Sizes, dtypes, alignment (16 bytes), scale, overlap rules and errors as for attn_fwd;
 * B * H <= 65535. Nothing is allocated; the calls only enqueue work on cuda_stream.
 */
size_t attn_decode_workspace_bytes(int B, int H, int d, int num_splits); /* 0 if invalid */
/* A split count that gives the GPU of the current device about eight CTAs per SM with
 * splits of at least 256 keys (0 for invalid sizes). */
int attn_decode_splits(int B, int H, int Nk);
/* The partial record of every split (writes partials). */
attn_status attn_decode_partial(const void* q, const void* k, const void* v, float* partials,
                                int B, int H, int Nk, int d, attn_dtype dtype, float scale,
                                int num_splits, void* cuda_stream);
/* Joins the records of each slice (reads partials, writes o and lse). Also the merge step
 * for partial results computed elsewhere, e.g. over key ranges held by different
 * processes, as long as they use this record layout. */
attn_status attn_decode_merge(const float* partials, void* o, float* lse, int B, int H, int d,
                              attn_dtype dtype, int num_splits, void* cuda_stream);
/* attn_decode_partial followed by attn_decode_merge on the same stream. */
attn_status attn_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                        float* partials, int B, int H, int Nk, int d, attn_dtype dtype,
                        float scale, int num_splits, void* cuda_stream);

/* attn_status_str - static, NUL-terminated name of a status code. */
const char* attn_status_str(attn_status s);

/*
 * attn_last_kernel_status - reads (with a blocking device-to-host copy on
 * cuda_stream, after the work queued before it) and clears the status word the
 * kernels set when a bounded pipeline wait runs out or a packed batch holds a
 * malformed sequence. Returns ATTN_OK when nothing was recorded since the last call,
 * ATTN_ERR_INVALID_ARG for a malformed sequence (code 0x7E), ATTN_ERR_TIMEOUT for a
 * wait, ATTN_ERR_CUDA if the copy fails. *where (may be NULL) receives the first code.
 * The status words are process-wide (one per device, per kernel file), not per call or
 * per stream: after calls on several streams or threads whose work overlapped, the word
 * holds the first code any of them recorded, and reading it clears it for all of them.
 */
attn_status attn_last_kernel_status(void* cuda_stream, int* where);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
