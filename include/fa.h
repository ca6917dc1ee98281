/*
 * fa.h — C ABI of the GB300 (sm_103a) exact attention forward library.
 *
 * What the library computes, for every batch b, head h and query row i:
 *
 *     s_j   = scale * (Q[b,h,i,:] . K[b,h,j,:])            for visible keys j
 *     O[b,h,i,:] = sum_j softmax(s)_j * V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_j exp(s_j)
 *
 * i.e. O = softmax(scale * Q K^T + mask) V, computed exactly (no
 * approximation of the softmax) without ever forming the score matrix in
 * device memory:
 *   - the definition: "Warmup Guide — Inference Optimization at Depth",
 *     Chapter 1 (S = Q K^T, P = softmax(S), O = P V) and Chapter 2 (safe
 *     softmax);
 *   - the tiled forward with the online softmax, each query block held on
 *     chip while K/V blocks stream through, O divided by the running sum
 *     once and written once: same page, Chapters 3 and 4, and
 *     "FlashAttention, speculative decoding, quantisation and parallelism",
 *     Mechanics;
 *   - the per-row statistics kept for the backward pass (Chapter 4), written
 *     as LSE = m + ln(l);
 *   - the decode-shaped path (few queries against a long KV cache, e.g. the
 *     k+1 positions of a speculative-decoding verify step): split the keys
 *     across CTAs and combine the partials, "Lecture 06 — Making Decode
 *     Fast", section 5 (Flash-Decoding).
 *
 * Conventions shared by every entry point
 *   Layout    Q, O: [B, H, Sq, d]; K, V: [B, H, Sk, d]; all contiguous,
 *             row-major, bf16 (IEEE bfloat16 bit patterns). LSE: [B, H, Sq]
 *             fp32, natural log, in units of the scaled logits.
 *   Causal    causal != 0 hides key j from query i unless
 *             j <= i + (Sk - Sq) (bottom-right alignment: the Sq queries sit
 *             after the first Sk - Sq keys). A row with no visible key gets
 *             O = 0 and LSE = -inf.
 *   Scale     any finite value (normally 1/sqrt(d)); the pages make it a
 *             plain factor of the scores. Zero gives uniform weights over
 *             the visible keys (O = their mean, LSE = ln of their count); a
 *             negative scale favours the least similar keys. The kernels
 *             form the scores with -Q when scale < 0 (the tensor-core
 *             operand negation, exact) and run the softmax with |scale|; at
 *             scale 0 they form them with a zero Q (every score is 0) and a
 *             softmax factor of 1. The scaled logits are fp32 values, so
 *             |scale * q . k| must stay within the fp32 range.
 *   Sizes     B, H, Sq, Sk >= 1; d in {64, 128}; Sq, Sk < 2^31; B*H < 2^31.
 *   Pointers  device pointers owned by the caller, 16-byte aligned (the
 *             kernels move tiles with TMA, which needs 16-byte aligned
 *             bases). The library never frees or retains them.
 *   Stream    a cudaStream_t passed as void* (NULL = legacy default stream).
 *             Every call enqueues work on it and returns without a host
 *             synchronisation, unless stated otherwise.
 *   Device    the current CUDA device of the calling thread; pointers must
 *             belong to it. The kernels need sm_103 (GB300).
 *   Errors    argument checks run first and return before anything is
 *             enqueued. A failed launch returns FA_ERR_CUDA. A bounded
 *             device-side wait that runs out sets a status word in device
 *             memory; fa_device_status() reads it.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,  /* null pointer, size <= 0, non-finite scale, bad split count */
    FA_ERR_UNSUPPORTED = 2,  /* d not in {64,128}, misaligned pointer, no sm_103 device */
    FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or a launch failed */
    FA_ERR_TIMEOUT = 4,      /* a kernel's bounded wait ran out (reported by fa_device_status) */
    FA_ERR_WORKSPACE = 5,    /* workspace missing or smaller than fa_workspace_size() */
    FA_ERR_BOUNDS = 6        /* a debug build's index check failed (reported by fa_device_status) */
} fa_status_t;

/*
 * Attention forward, dispatching on the shape:
 *   Sq <= FA_VERIFY_MAX_SQ : the split-KV path (fa_verify_forward) with an
 *                            automatic split count; its workspace is taken
 *                            from a library-owned stream-ordered memory pool
 *                            (cudaMallocFromPoolAsync / cudaFreeAsync on
 *                            `stream`) that keeps freed blocks for the next
 *                            call, so it holds the largest workspace a call
 *                            has needed until the process exits;
 *   otherwise              : the tiled prefill path (fa_prefill_forward),
 *                            which needs no workspace.
 * q, k, v: inputs; o, lse: outputs (every element of both is written).
 */
fa_status_t fa_forward(const void *q, const void *k, const void *v, void *o, float *lse,
                       int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal,
                       float scale, void *stream);

/* Largest Sq that fa_forward sends to the split-KV path. */
#define FA_VERIFY_MAX_SQ 16

/*
 * Bytes of workspace fa_forward_ws needs for this shape (0 when the shape
 * takes the prefill path). The split-KV size depends on the current device's
 * SM count; returns 0 for invalid sizes or when no device can be queried.
 */
size_t fa_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d);

/*
 * Same as fa_forward, but never allocates: the split-KV path uses the
 * caller's `workspace` (device memory, 256-byte aligned, at least
 * fa_workspace_size() bytes, not used concurrently by another call).
 * Returns FA_ERR_WORKSPACE if it is missing or too small.
 */
fa_status_t fa_forward_ws(const void *q, const void *k, const void *v, void *o, float *lse,
                          int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal,
                          float scale, void *workspace, size_t ws_bytes, void *stream);

/*
 * The tiled prefill kernel for any Sq (the pages' FlashAttention forward):
 * each CTA keeps two 128-row query tiles on chip (tensor memory for S and O),
 * streams 128-key K/V tiles through a TMA-fed shared-memory ring, forms
 * S = Q K^T with tcgen05 MMAs, applies the online softmax, accumulates
 * O += P V with tcgen05 MMAs, skips key tiles above the causal diagonal, and
 * writes O / l and LSE once. No workspace.
 * The kernel is persistent (one CTA per SM) and takes its work items from a
 * library-owned counter in device memory. Launches use the library's 1024
 * counters in turn, and each launch returns its counter to zero, so up to
 * 1024 launches may run at the same time; a 1025th running together with
 * the one that took the same counter would share it.
 */
fa_status_t fa_prefill_forward(const void *q, const void *k, const void *v, void *o, float *lse,
                               int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d,
                               int causal, float scale, void *stream);

/*
 * The FP8 forward: the FlashAttention-3 variant with 8-bit float inputs that
 * "FlashAttention, speculative decoding, quantisation and parallelism" (The
 * problem it solves) and "Lecture 06 — Making Decode Fast" (section 5) name.
 * The pages give no format or recipe; this entry point takes:
 *   q         E4M3 bytes [B, H, Sq, 128], row-major (OCP E4M3: bias 7, no
 *             infinities, 0x7F/0xFF NaN; finite values up to 448);
 *   k, v      E4M3 bytes [B, H, Sk, 128];
 *   o         bf16 [B, H, Sq, 128] out;  lse  fp32 [B, H, Sq] out;
 *   q_descale, k_descale, v_descale
 *             one fp32 per tensor: a byte stands for descale * its E4M3 value.
 * It computes, per row, the scores s_j = scale * q_descale * k_descale *
 * (q . k_j) accumulated in fp32 on the FP8 tensor cores, the online softmax
 * with an integer reference M in log2 units, weights 2^(s_j log2 e - M)
 * scaled by 2^4 and rounded to E4M3 (nearest, ties to even) before O += P V
 * runs on the FP8 tensor cores, the row sum l taken before that rounding,
 * then o = v_descale * O / l and lse = ln(sum_j e^(s_j)) (natural log; -inf
 * and o = 0 for a row with no visible key). M is an integer that trails the
 * row's running max by less than 4.8, so against the row's final max the
 * weights are rounded at a scale of 2^4 to 2^9: every weight of at least
 * 2^-10 of the row max gets the value the scale 2^7 gives (up to an exact
 * power of two); smaller ones may round on E4M3's subnormal grid (at most
 * 2^-12 of the row's largest weight each). Causal masking is bottom-right as
 * in fa_forward.
 * d must be 128; q, k, v, o 16-byte aligned, lse 4-byte aligned; any
 * Sq, Sk >= 1. The caller owns every buffer; nothing is allocated.
 * scale: any finite value, as in fa_forward; the descales must be > 0.
 * Errors: FA_ERR_INVALID_ARG for null pointers, sizes <= 0, a non-finite
 * scale or descale; FA_ERR_UNSUPPORTED for d != 128, a descale <= 0, a
 * product |scale| * q_descale * k_descale beyond the fp32 range, misaligned
 * pointers or a device other than sm_103.
 */
fa_status_t fa_forward_fp8(const void *q, const void *k, const void *v, void *o, float *lse,
                           int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal,
                           float scale, float q_descale, float k_descale, float v_descale,
                           void *stream);

/*
 * The decode-shaped split-KV kernel (Flash-Decoding) for 1 <= Sq <= 16:
 * the keys of each (b, h) are cut into n_split contiguous chunks, one CTA
 * per (chunk, b, h) computes a partial (O_s, LSE_s), and a combine kernel
 * merges the partials with LSE weights:
 *     LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s.
 * n_split = 0 picks a count that fills the GPU; otherwise 1 <= n_split <=
 * ceil(Sk / 64) (chunks are multiples of 64 keys). With one chunk the
 * partial is the result and no workspace is needed.
 * Returns FA_ERR_UNSUPPORTED for Sq > 16.
 */
fa_status_t fa_verify_forward(const void *q, const void *k, const void *v, void *o, float *lse,
                              int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d,
                              int causal, float scale, int n_split, void *workspace,
                              size_t ws_bytes, void *stream);

/*
 * Workspace bytes fa_verify_forward needs for this shape and split count
 * (n_split = 0: the automatic count on the current device, which needs a
 * CUDA device to query; returns 0 when none is present). Layout of the
 * workspace: partial O_s as fp32 [n_split, B, H, Sq, d], then LSE_s as fp32
 * [n_split, B, H, Sq], each part 256-byte aligned.
 */
size_t fa_verify_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d,
                                int n_split);

/* The split count fa_verify_forward uses for n_split = 0 on the current device (0 on error). */
int fa_verify_auto_splits(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d);

/*
 * Split-KV verify with a tree of draft tokens: the Sq queries are candidate
 * tokens of a draft tree appended after Sk - Sq cached keys; each candidate
 * attends to the whole cache and to the candidates its tree mask selects
 * (normally its ancestors and itself), so several continuations are verified
 * in one pass ("Lecture 06 — Making Decode Fast", section 3: tree-attention
 * over a draft tree).
 *   tree_mask : device uint32 [B, Sq]; bit k of tree_mask[b][i] set means
 *               query i of sequence b sees key Sk - Sq + k (bits >= Sq are
 *               ignored). A chain (bits 0..i) is the causal case.
 * Other arguments as fa_verify_forward (causal is replaced by the mask).
 * Returns FA_ERR_INVALID_ARG for a NULL or misaligned tree_mask.
 */
fa_status_t fa_verify_tree_forward(const void *q, const void *k, const void *v, void *o,
                                   float *lse, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                                   int64_t d, const uint32_t *tree_mask, float scale, int n_split,
                                   void *workspace, size_t ws_bytes, void *stream);

/*
 * Split-KV verify reading K and V through a block table (paged KV cache,
 * "Warmup Guide — Inference Optimization at Depth", Chapter 8 and its Q&A:
 * the kernel walks the block table once per tile). Sequences may have
 * different lengths.
 *   k_pages, v_pages : device bf16 [num_pages, H, page_size, d] page pools.
 *   block_table      : device int32 [B, max_pages_per_seq]; entry p of row b
 *                      is the pool page holding keys [p*page_size,
 *                      (p+1)*page_size) of sequence b. Entries past a
 *                      sequence's length are not read.
 *   seq_lens         : device int32 [B], the keys of each sequence; values are
 *                      clamped to [0, max_pages_per_seq * page_size]. A
 *                      sequence's last Sq keys are its draft positions.
 *   page_size        : 16, 32, or a multiple of 64 (one TMA box per page per
 *                      64-key stage, or per page when pages are smaller).
 *   max_seq_len      : host value, >= every seq_lens entry and
 *                      <= max_pages_per_seq * page_size; sets the split size.
 *   causal, tree_mask: bottom-right causal per sequence, or (tree_mask != NULL)
 *                      the tree masks of fa_verify_tree_forward.
 *   workspace        : fa_verify_workspace_size(B, H, Sq, max_seq_len, d,
 *                      n_split) bytes when the split count exceeds one.
 * A page index outside [0, num_pages) is read as zeros (it never faults).
 * q, o, lse as fa_verify_forward.
 */
fa_status_t fa_verify_paged_forward(const void *q, const void *k_pages, const void *v_pages,
                                    const int32_t *block_table, const int32_t *seq_lens, void *o,
                                    float *lse, int64_t B, int64_t H, int64_t Sq, int64_t d,
                                    int64_t num_pages, int64_t page_size,
                                    int64_t max_pages_per_seq, int64_t max_seq_len, int causal,
                                    const uint32_t *tree_mask, float scale, int n_split,
                                    void *workspace, size_t ws_bytes, void *stream);

/*
 * Backward pass of the attention forward (prefill path): given the forward's
 * inputs, its outputs O and LSE, and the upstream gradient dO, writes dQ, dK,
 * dV. P is never stored: its tiles are recomputed from Q, K and LSE
 * ("Warmup Guide — Inference Optimization at Depth", Chapter 4), i.e.
 *     P = exp(scale * Q K^T - LSE) (masked),  D_i = dO_i . O_i,
 *     dV = P^T dO,  dS = P o (dO V^T - D),  dK = scale * dS^T Q,
 *     dQ = scale * dS K.
 *   q, k, v, o, lse, causal, scale : as passed to / returned by fa_forward.
 *   dout      : device bf16 [B, H, Sq, d].
 *   dq        : device bf16 [B, H, Sq, d];  dk, dv: device bf16 [B, H, Sk, d].
 *   workspace : fa_backward_workspace_size() bytes of device memory
 *               (scratch: -D and -LSE * log2(e) per padded query row),
 *               256-byte aligned; NULL takes it from the library's
 *               stream-ordered pool on `stream` (as fa_forward does).
 * Enqueues three kernels on `stream`. The third (dQ) is launched with
 * programmatic stream serialization so that it starts on the SMs the second
 * (dK, dV) leaves idle; it waits for the second before completing, so the
 * call as a whole is ordered on `stream` like any other (also under CUDA
 * graph capture). Rows with no visible key contribute nothing. Same shape
 * limits and errors as fa_prefill_forward.
 */
fa_status_t fa_backward(const void *q, const void *k, const void *v, const void *o,
                        const float *lse, const void *dout, void *dq, void *dk, void *dv,
                        int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal,
                        float scale, void *workspace, size_t ws_bytes, void *stream);

/* Workspace bytes fa_backward needs (0 for invalid sizes). */
size_t fa_backward_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d);

/*
 * Attention forward on HOST-resident tensors, with the transfers inside the
 * call: the end-to-end form of fa_forward for a caller whose Q, K, V live in
 * host memory and who wants O and LSE back in host memory.
 *   q, k, v, o, lse : host pointers, same layouts as fa_forward. Page-locked
 *                     memory (cudaHostAlloc / cudaHostRegister) lets the
 *                     copies run asynchronously and overlap; pageable memory
 *                     works but serialises them.
 *   workspace       : device memory of at least fa_forward_host_workspace_size
 *                     bytes, 256-byte aligned, used to stage Q, K, V, O, LSE
 *                     (and split-KV partials); NULL makes the call take it from
 *                     the stream-ordered allocator on `stream`.
 * The (b, h) pairs are processed in FA_HOST_CHUNKS consecutive groups: the
 * host-to-device copies of group c+1 overlap the kernels of group c and the
 * device-to-host copies of group c-1, on copy and compute streams owned by
 * the library. When o is pinned host memory mapped into the device's address
 * space (cudaHostAlloc / cudaHostRegister under unified addressing) and
 * 16-byte aligned, O returns through stores by a few CTAs of the library,
 * which leave the host link to the input copies; otherwise, and for lse,
 * through cudaMemcpyAsync. All of it is ordered after work already queued on `stream`,
 * and `stream` waits for all of it, so synchronising `stream` (or an event
 * recorded on it afterwards) means o and lse are filled. Calls from several
 * host threads are serialised on the library's streams.
 * Errors as fa_forward; a NULL host pointer is FA_ERR_INVALID_ARG.
 */
fa_status_t fa_forward_host(const void *q, const void *k, const void *v, void *o, float *lse,
                            int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal,
                            float scale, void *workspace, size_t ws_bytes, void *stream);

/* Number of (b, h) groups fa_forward_host pipelines (fewer if B*H is smaller). */
#define FA_HOST_CHUNKS 16

/*
 * Device workspace bytes fa_forward_host needs for this shape (device copies of
 * Q, K, V, O, LSE plus, for Sq <= FA_VERIFY_MAX_SQ, the split-KV partials of
 * one group on the current device). 0 for invalid sizes or without a device.
 */
size_t fa_forward_host_workspace_size(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d);

/*
 * Size of the library-owned scratch used by fa_verify_forward_static.
 */
#define FA_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * fa_verify_forward without any allocation and without a caller workspace.
 * The pages have no counterpart: it exists for callers that cannot call
 * cudaMalloc (plugins in a host runtime that owns all device memory and
 * passes them only their input and output buffers; serving loops that
 * reserved nearly all of HBM up front; loops that cannot accept the
 * synchronisation an allocation may cause).
 * Arguments, layouts, checks and results are those of fa_verify_forward; the
 * argument checks come first, with the same codes. The split-KV partials go
 * to a file-scope device array of FA_STATIC_SCRATCH_BYTES bytes that every
 * GPU loading the library holds until exit. n_split = 0 takes the automatic
 * count, lowered if need be to the largest count whose partials
 * (fa_verify_workspace_size) fit in the array; one split needs none, so
 * every shape fa_verify_forward accepts runs. An explicit n_split whose
 * partials exceed FA_STATIC_SCRATCH_BYTES returns FA_ERR_WORKSPACE.
 * The first call on a device looks up the array's address with the device
 * current; make it before any stream capture. The address is kept for the
 * calling thread's CUDA context: after cudaDeviceReset (or under another
 * driver context) the next call looks it up again. All calls share the array
 * and it keeps the last call's contents: calls that overlap on the GPU race.
 */
fa_status_t fa_verify_forward_static(const void *q, const void *k, const void *v, void *o,
                                     float *lse, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                                     int64_t d, int causal, float scale, int n_split,
                                     void *stream);

/* Static text for a status code. */
const char *fa_status_string(fa_status_t status);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device: FA_OK; FA_ERR_BOUNDS if, in a library built
 * with FA_DEBUG (device-side index checks; see fa_testing.h), a check failed
 * since the last call (the access was skipped); else FA_ERR_TIMEOUT if a
 * kernel gave up on a bounded wait since the last call (its outputs are then
 * undefined). Returns FA_ERR_CUDA if the synchronisation itself fails.
 */
fa_status_t fa_device_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
