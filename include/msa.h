/*
 * msa.h - C ABI of the MSA (MiniMax-style sparse attention) training library for GB300 (sm_103a).
 *
 * One training step of MSA with grouped-query attention (GQA) over a packed
 * batch of variable-length documents:
 *
 *   msa_proxy_select  proxy scores q_p . k_p^T for every causal key, max-pooled
 *                     over 128-token KV blocks, and per query token the top-k
 *                     blocks with its own (diagonal) block always kept.
 *                     Block selection by the maximum proxy score inside each
 *                     128-token block: "Dramatically Speeding Up Million-Token
 *                     Training! ... 'Flash-MSA' ..." (ai-minor.com), section
 *                     "What's Happening? News Overview"; proxy heads managing KV
 *                     subsets: Flash-MSA summary (socker-news.uzaya.net), 要約.
 *   msa_fwd           exact softmax attention of every query head over the
 *                     selected blocks of its KV group (GQA: same page, News
 *                     Overview), computed block by block with the queries
 *                     regrouped per KV block (the "MoBA varlen trick" of the
 *                     Flash-MSA summary) and merged by log-sum-exp.
 *   msa_bwd           dQ/dK/dV of the attention and, fused into the same pass,
 *                     the gradient of the proxy training loss ("... 'Flash-MSA'
 *                     ...", section "Why Does This Matter?", fused backward).
 *
 * The pages do not define the proxy's training signal.  This library uses
 *   KL_{t,g} = sum_{b in Sel} m_b (log m_b - log p_b),
 *   p_b = softmax over the selected blocks of the pooled proxy scores S_b,
 *   m_b = (1/G) sum over the group's G heads of the attention probability mass
 *         inside block b (treated as a constant target),
 * and the loss kl_weight * sum_{t,g} KL_{t,g}.
 *
 * Block pattern (window w, dilation s): besides the diagonal, the blocks
 * j - s*u for u = 1..w (those >= 0) are always kept; they take w of the k
 * slots and the top-k choice fills the remaining k-1-w from the other earlier
 * blocks (all of them when they fit).  w = 0 is the plain rule.  The pattern
 * is configurable by window size and dilation ("Flash-MSA: Ein Training mit
 * einer Million Tokens ohne hohe Rechenkosten", keelcrux.com, section "Under
 * the hood"); the set above is this library's reading of those two words.
 * With w = k-1 and s = 1 the selection is a sliding window of k blocks.
 *
 * Notation: T total tokens, Hq query heads, Hkv KV heads (groups), G = Hq/Hkv,
 * d head dim, dp proxy dim, B = 128 block size, K = top_k (diagonal included).
 * A token at doc-local position i lies in block j = i / B.  Blocks restart at
 * every document start; block ids below are doc-local.
 *
 * Layouts (all row-major, packed over documents, token-major):
 *   q, dO, o          [T, Hq, d]     bf16 (raw bits in uint16_t)
 *   k, v              [T, Hkv, d]    bf16
 *   q_p, k_p          [T, Hkv, dp]   bf16
 *   cu_seqlens        [num_docs + 1] int32, cu_seqlens[0] = 0, non-decreasing,
 *                                    cu_seqlens[num_docs] = T
 *   sel_idx           [T, Hkv, K]    int32 selected doc-local block ids,
 *                                    ascending, diagonal last, -1 padded
 *   sel_score         [T, Hkv, K]    fp32 pooled proxy score S_b (0 for padding)
 *   sel_arg           [T, Hkv, K]    uint8 offset inside the block of the key
 *                                    attaining S_b (lowest such key)
 *   plse              [T, Hkv]       fp32 logsumexp of S_b over the selection
 *   tie               [T, Hkv]       uint8 1 when the last candidate the top-k
 *                                    choice takes and the first it leaves
 *                                    (always-kept blocks are not candidates)
 *                                    differ in score by less than 1e-3
 *   o_res             [T, Hq, d]     bf16 rounding residual of o: bf16(O - o) for the
 *                                    fp32 result O, so o + o_res carries ~16
 *                                    mantissa bits (saved for msa_bwd, whose
 *                                    D = rowsum(dO * O) needs more than bf16 o)
 *   lse               [T, Hq]        fp32 natural-log softmax normaliser
 *   mass              [T, Hkv, K]    fp32 target mass m_b per selected block
 *   dq                [T, Hq, d]     fp32;  dk, dv [T, Hkv, d] fp32
 *   dq_p, dk_p        [T, Hkv, dp]   fp32
 *   kl_loss           one fp64 on the device
 *
 * Conventions:
 *   - The caller owns every buffer (inputs, outputs, workspace); the library
 *     never allocates device memory and keeps no per-call state.  Query the
 *     workspace size with the *_workspace_size functions; the workspace needs
 *     no initialisation.
 *   - Every pointer argument is a device pointer aligned to 16 bytes unless
 *     stated otherwise.  params is a host pointer.
 *   - All calls are asynchronous on `stream` and may be captured in a CUDA
 *     graph.  Argument checks on the host return an error before any launch.
 *   - Supported shapes: d in {64, 128}, dp in {32, 64}, block = 128,
 *     G in {1, 2, 4, 8}, 1 <= top_k <= 16, T < 2^27, and at most 49152 KV
 *     blocks in the batch; anything else returns MSA_ERR_UNSUPPORTED.  There is
 *     no CPU fallback.
 *   - Errors found on the device (malformed cu_seqlens, an internal wait that
 *     ran out) are recorded in a device status word; read it with
 *     msa_get_device_status after the stream has reached the call.  Its
 *     address is looked up once per device and cached for the life of the
 *     process, so the library must not be used after cudaDeviceReset.
 *   - Batches of more than 2048 KV blocks run the forward and backward block
 *     kernels in query chunks of 2048 blocks (this bounds the workspace).  The
 *     environment variable MSA_QUERY_CHUNK_BLOCKS, read at every call, sets a
 *     smaller positive chunk (in KV blocks) instead; it exists so that tests
 *     can take the chunked path on small batches, and results do not depend
 *     on it beyond fp32 rounding of dk, dv and dk_p (summed chunk by chunk).
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* msa_stream_t;

typedef struct msa_params {
  int32_t total_tokens; /* T */
  int32_t num_docs;     /* documents in the packed batch */
  int32_t max_seqlen;   /* upper bound of any document length (host-known) */
  int32_t hq, hkv;      /* query heads, KV heads; hq % hkv == 0 */
  int32_t d, dp;        /* head dim, proxy dim */
  int32_t block;        /* KV block size; must be 128 */
  int32_t top_k;        /* selected blocks per (token, group), diagonal included */
  int32_t window;       /* block pattern: always-kept earlier blocks, 0 <= window <= top_k - 1
                           (0: none; see "Block pattern" above) */
  int32_t dilation;     /* block pattern: spacing of those blocks, >= 0 (0 is read as 1) */
  float softmax_scale;  /* multiplies q . k (1.0 when q is pre-scaled) */
  float proxy_scale;    /* multiplies q_p . k_p (1.0 when q_p is pre-scaled) */
  float kl_weight;      /* lambda of the proxy KL loss */
  uint32_t flags;       /* MSA_FLAG_REUSE_REGROUP, MSA_FLAG_TEST_STALL_SELECT or 0; other bits
                           are rejected */
} msa_params;

/*
 * msa_fwd and msa_bwd: the workspace passed to the call is the one the
 * preceding msa_proxy_select or msa_fwd call used, on the same stream, with
 * the same params, cu_seqlens and sel_idx, and nothing has written to it
 * since.  The call then reuses the block lists (queries regrouped per KV
 * block) left at the front of the workspace instead of rebuilding them (5
 * fewer kernel launches).  All three workspace layouts share that prefix.
 * msa_proxy_select ignores the flag.  msa_proxy_select_noalloc has no
 * workspace and builds no block lists, so the flag must not be set on a call
 * whose preceding call was msa_proxy_select_noalloc.  If the condition does
 * not hold, the results are undefined.
 */
#define MSA_FLAG_REUSE_REGROUP 0x1u

/*
 * Test hook for the failure path (no use in training).  msa_proxy_select's
 * scoring kernel withholds the load of its query tile, so the wait of its MMA
 * warp on that load (or the epilogue's wait on the first scores, whichever
 * gives up first) runs out after the bounded-wait limit (about half a second
 * of SM cycles).  Every CTA then records MSA_ERR_TIMEOUT in the device status
 * word (kernel 1, see msa_last_status_word), lets the copies it did issue
 * land, frees its tensor memory and returns without writing its outputs:
 * sel_idx, sel_score, plse and tie keep their previous contents, and the rest
 * of the call (block lists, argmax offsets) runs on them.  The GPU stays
 * usable; the next call without the flag is unaffected.  msa_fwd and msa_bwd
 * ignore the flag.
 */
#define MSA_FLAG_TEST_STALL_SELECT 0x100u

typedef enum msa_status {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, inconsistent sizes */
  MSA_ERR_UNSUPPORTED = 2, /* shape outside the supported set */
  MSA_ERR_WORKSPACE = 3,   /* workspace smaller than *_workspace_size() */
  MSA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  MSA_ERR_TIMEOUT = 5,     /* device: a bounded wait inside a kernel ran out */
  MSA_ERR_DEVICE_CHECK = 6 /* device: malformed cu_seqlens or index found in a kernel */
} msa_status;

/* Workspace bytes each call needs for these params (0 if params are invalid). */
size_t msa_select_workspace_size(const msa_params* params);
size_t msa_fwd_workspace_size(const msa_params* params);
size_t msa_bwd_workspace_size(const msa_params* params);

/*
 * Proxy scoring, 128-key block max-pool and top-k block selection.
 * Inputs: cu_seqlens, q_p, k_p.  Outputs: sel_idx, sel_score, sel_arg, plse, tie.
 * The [T, T] score matrix and the [T, blocks] pooled matrix are never stored.
 * The argmax of each chosen earlier block is found after the selection, from
 * the block lists (queries regrouped per KV block) that the call leaves at the
 * front of the workspace for msa_fwd (see MSA_FLAG_REUSE_REGROUP).
 */
msa_status msa_proxy_select(const msa_params* params, const int32_t* cu_seqlens,
                            const uint16_t* q_p, const uint16_t* k_p, int32_t* sel_idx,
                            float* sel_score, uint8_t* sel_arg, float* plse, uint8_t* tie,
                            void* workspace, size_t workspace_bytes, msa_stream_t stream);

/*
 * Attention over the selected blocks.  Inputs: cu_seqlens, q, k, v, sel_idx.
 * Outputs: o (bf16), and saved for msa_bwd: o_res, lse, and mass, the per-block
 * target of the proxy loss.
 */
msa_status msa_fwd(const msa_params* params, const int32_t* cu_seqlens, const uint16_t* q,
                   const uint16_t* k, const uint16_t* v, const int32_t* sel_idx, uint16_t* o,
                   uint16_t* o_res, float* lse, float* mass, void* workspace,
                   size_t workspace_bytes, msa_stream_t stream);

/*
 * Backward of sum(o * dO) + kl_weight * sum KL.  Inputs: the forward's inputs and
 * outputs, dO, and the selection.  Outputs (all overwritten, no accumulation):
 * dq, dk, dv, dq_p, dk_p and the scalar kl_loss.  The selection is held
 * constant (it is discrete); the target mass receives no gradient.  With
 * MSA_FLAG_REUSE_REGROUP in params->flags the block lists msa_fwd built in the
 * same workspace are reused (see the flag).
 */
msa_status msa_bwd(const msa_params* params, const int32_t* cu_seqlens, const uint16_t* q,
                   const uint16_t* k, const uint16_t* v, const uint16_t* q_p, const uint16_t* k_p,
                   const uint16_t* o, const uint16_t* o_res, const float* lse, const float* mass,
                   const uint16_t* dO,
                   const int32_t* sel_idx, const float* sel_score, const uint8_t* sel_arg,
                   const float* plse, float* dq, float* dk, float* dv, float* dq_p, float* dk_p,
                   double* kl_loss, void* workspace, size_t workspace_bytes, msa_stream_t stream);

/*
 * msa_proxy_select without a workspace, for callers that cannot allocate
 * device memory.  Some host programs have no way to hand the library a
 * buffer: all device memory belongs to another component's allocator that
 * exposes no raw pointers, or the call sits on a path where cudaMalloc (which
 * can synchronise the whole device) is not allowed.  This entry point takes
 * the same inputs and writes the same outputs as msa_proxy_select; its only
 * scratch, the per-document block prefix, lives in a static device array of
 * 16384 int32 (64 KB) that every GPU loading the library keeps until the
 * process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.  Limits and caveats:
 *   - batches of more than 16382 documents return MSA_ERR_WORKSPACE;
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, so make that first
 *     call before any stream capture;
 *   - all calls share the one array: calls that overlap on the GPU (for
 *     example on two streams without ordering between them) race on it.
 *     Each call writes every entry it reads, so no clearing is needed;
 *   - it leaves no block lists anywhere, so a following msa_fwd or msa_bwd
 *     must not set MSA_FLAG_REUSE_REGROUP (it builds its own lists instead);
 *   - the array's address is cached per device for the life of the process:
 *     after cudaDeviceReset (or any teardown of the device's primary context)
 *     the library must not be called again in that process.  The same holds
 *     for the device status word every entry point uses.
 * The pages have no counterpart of this entry point.
 */
msa_status msa_proxy_select_noalloc(const msa_params* params, const int32_t* cu_seqlens,
                                    const uint16_t* q_p, const uint16_t* k_p, int32_t* sel_idx,
                                    float* sel_score, uint8_t* sel_arg, float* plse, uint8_t* tie,
                                    msa_stream_t stream);

/*
 * Synchronises `stream`, returns the device status word of the current device
 * (MSA_OK, MSA_ERR_TIMEOUT or MSA_ERR_DEVICE_CHECK; the first error recorded
 * wins) and resets it to MSA_OK.  Returns MSA_ERR_CUDA if the stream itself
 * reports an error.
 */
msa_status msa_get_device_status(msa_stream_t stream);

/*
 * Full device status word seen by the last msa_get_device_status call on the
 * calling host thread.  Bits 0-7 hold the status code.  For MSA_ERR_TIMEOUT,
 * bits 8-11 name the kernel whose wait ran out (1 proxy select, 2 forward,
 * 3 backward), bits 12-19 the barrier index inside it and bits 20-31 the tile
 * (or key block) it was working on, saturated at 4095.
 */
uint32_t msa_last_status_word(void);

/*
 * Number of CUDA kernels this library has launched in this process (all
 * devices and threads), for accounting in benchmarks.
 */
uint64_t msa_launch_count(void);

/*
 * Opt-in timing hook.  While set, every launch of the named kernel records
 * `start` on the call's stream right before it and `stop` right after it
 * (`start`/`stop` are cudaEvent_t handles owned by the caller; pass null to
 * clear).  which: 1 proxy scoring + selection kernel, 2 forward block kernel,
 * 3 backward block kernel.  A batch of more than 2048 KV blocks runs the
 * forward and backward block kernels once per query chunk; `start` is then
 * recorded before the first of them and `stop` after the last, so the span
 * includes the merge / reduce passes of the earlier chunks in between.
 * Process-global; not for concurrent use from several threads.  Returns
 * MSA_ERR_INVALID_ARG for an unknown `which`.
 */
typedef struct CUevent_st* msa_event_t;
msa_status msa_set_profile_events(int which, msa_event_t start, msa_event_t stop);

/* Static, human-readable name of a status code. */
const char* msa_status_string(msa_status status);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
