/*
 * dflash.h - C ABI of the GB300 (sm_103a) greedy block-diffusion speculative
 * decoding round: target prefill, block drafting with target-context KV
 * injection, one-pass target verification, greedy acceptance and rollback.
 *
 * The operations follow two public pages:
 *   [digest] "DFlash: Block Diffusion for Flash Speculative Decoding"
 *            (paper digest: Method / Inference §4.1, the greedy decoding-round
 *            and draft-layer pseudocode, "Paper vs code").
 *   [review] "DFlash: Why a Diffusion Drafter Can Accelerate an Autoregressive
 *            Model" (technical review: §2.3 eq. 2, §4.1, Algorithm 1,
 *            §5.1 eq. 9-10).
 * and, for the runtime block size only, the "DFlash" wiki page (Ablations).
 *
 * Conventions
 * -----------
 * - Matrices are row-major [out_features, in_features] (y = W x), element
 *   type given by dflash_config.dtype (fp32 or bf16).  Norm scales are fp32.
 * - Every call is ordered on the CUDA stream given to dflash_init.  A call
 *   whose outputs are host pointers returns after the results are on the host;
 *   a call whose outputs are device pointers returns without synchronising.
 * - Token arrays may be host or device memory; the library asks the CUDA
 *   runtime which one a pointer is.
 * - No call throws, aborts or traps.  Each returns a dflash_status; the text
 *   of the last failure is available from dflash_last_error.  A call that
 *   fails a precondition changes no state.
 * - Device-side checks (for example a token id outside [0, vocab) passed in
 *   device memory) never fault: they record an error word that the next
 *   synchronising call turns into DFLASH_E_DEVICE_CHECK.
 * - One session serves one host thread at a time (calls on a ctx must not
 *   overlap); separate sessions are independent and may be driven from
 *   different threads.  dflash_init's error text is kept per thread.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DFLASH_OK = 0,
    DFLASH_E_INVAL = 1,        /* bad argument or inconsistent configuration */
    DFLASH_E_NOMEM = 2,        /* a device allocation failed */
    DFLASH_E_CUDA = 3,         /* a CUDA runtime call failed */
    DFLASH_E_STATE = 4,        /* call out of order (verify before draft, draft before prefill, ...) */
    DFLASH_E_CAPACITY = 5,     /* a sequence would grow past max_seq_len, or the KV page pool is full */
    DFLASH_E_TIMEOUT = 6,      /* a bounded device-side wait ran out */
    DFLASH_E_DEVICE_CHECK = 7  /* a device-side argument check failed */
} dflash_status;

enum { DFLASH_DTYPE_F32 = 0, DFLASH_DTYPE_BF16 = 1 };

/* Flags (dflash_config.flags). */
enum {
    DFLASH_FLAG_KEEP_LOGITS = 1, /* keep fp32 logits of the last prefill / draft / verify for dflash_inspect */
    DFLASH_FLAG_PROFILE = 2,     /* time every kernel class with CUDA events (see DFLASH_INSPECT_PROFILE) */
    DFLASH_FLAG_NO_GRAPHS = 4    /* launch every kernel directly instead of replaying captured CUDA graphs */
};

/* Kernel classes reported by DFLASH_INSPECT_PROFILE. */
enum {
    DFLASH_K_GEMM_QKV = 0,     /* fused q/k/v projection (target and draft layers) */
    DFLASH_K_GEMM_O = 1,       /* attention output projection + residual */
    DFLASH_K_GEMM_GATE_UP = 2, /* SwiGLU gate/up projection */
    DFLASH_K_GEMM_DOWN = 3,    /* SwiGLU down projection + residual */
    DFLASH_K_GEMM_HEAD = 4,    /* shared LM head */
    DFLASH_K_GEMM_FC = 5,      /* context fusion W_c */
    DFLASH_K_GEMM_CTX_KV = 6,  /* context key/value projection of the draft layers */
    DFLASH_K_ATTENTION = 7,
    DFLASH_K_NORM = 8,
    DFLASH_K_ROPE_STORE = 9,
    DFLASH_K_SWIGLU = 10,
    DFLASH_K_ARGMAX = 11,
    DFLASH_K_OTHER = 12,
    DFLASH_K_SAMPLING = 13,    /* filtered laws, draws and acceptance of the sampled round */
    DFLASH_K_COUNT = 14
};

/* One kernel class in the profile: launches, summed device time (CUDA events
 * bracketing each launch on the session stream), and the algorithmic bytes
 * moved and flops performed by those launches. */
typedef struct {
    int64_t launches;
    double ms;
    double bytes;
    double flops;
} dflash_profile_entry;

enum { DFLASH_MAX_CTX_LAYERS = 16 };

/* Device allocator used for every library-owned buffer.  Returns NULL on
 * failure.  When both are NULL the library uses cudaMalloc / cudaFree. */
typedef void* (*dflash_alloc_fn)(size_t bytes, void* user);
typedef void (*dflash_free_fn)(void* ptr, void* user);

typedef struct {
    int32_t dtype;             /* DFLASH_DTYPE_F32 or DFLASH_DTYPE_BF16 */
    int32_t vocab;             /* V */
    int32_t d_model;           /* d; multiple of 64 */
    int32_t n_heads;           /* H query heads */
    int32_t n_kv_heads;        /* H_kv; H % H_kv == 0 */
    int32_t head_dim;          /* 64 or 128 */
    int32_t ffn;               /* SwiGLU hidden size F; multiple of 64 */
    int32_t target_layers;     /* L_t */
    int32_t target_qk_norm;    /* 1: per-head RMSNorm of q and k in target layers */
    int32_t draft_layers;      /* L_d (the drafter always normalises q and k per head) */
    int32_t block_size;        /* B: anchor + B-1 mask positions; 1 <= B <= 32 */
    int32_t n_ctx_layers;      /* k target layers whose hidden states form the context feature */
    int32_t ctx_layer_ids[DFLASH_MAX_CTX_LAYERS]; /* 0-based target layers, residual after the layer */
    int32_t mask_token;        /* id embedded at the B-1 mask positions */
    int32_t max_batch;         /* sequences per session */
    int32_t max_seq_len;       /* longest sequence: prompt + generated + B */
    int32_t flags;             /* DFLASH_FLAG_* */
    float rms_eps;             /* RMSNorm epsilon */
    double rope_theta;         /* RoPE base */
    dflash_alloc_fn alloc;     /* optional allocator (see above) */
    dflash_free_fn free;
    void* alloc_user;
    int64_t kv_pool_tokens;    /* KV cache capacity shared by the batch, in tokens (rounded up to
                                  64-token pages); 0 = max_batch * max_seq_len */
} dflash_config;

/* One decoder layer, device pointers.  wq, wk, wv, w_gate and w_up are read
 * only inside dflash_init, which packs them into library-owned matrices (one
 * [q; k; v] projection, and in bf16 gate and up interleaved in 64-row tiles
 * for the fused SwiGLU), so they may be freed afterwards.  wo and w_down are
 * borrowed: every call reads them in place, so they must stay allocated and
 * unchanged until dflash_destroy, and be 16-byte aligned.  Norm scales are
 * copied. */
typedef struct {
    const void* wq;            /* [H*hd, d] */
    const void* wk;            /* [H_kv*hd, d] */
    const void* wv;            /* [H_kv*hd, d] */
    const void* wo;            /* [d, H*hd] */
    const void* w_gate;        /* [F, d] */
    const void* w_up;          /* [F, d] */
    const void* w_down;        /* [d, F] */
    const float* attn_norm;    /* [d] */
    const float* mlp_norm;     /* [d] */
    const float* q_norm;       /* [hd]; NULL for target layers without QK-norm */
    const float* k_norm;       /* [hd]; NULL for target layers without QK-norm */
} dflash_layer_weights;

/* Target decoder plus drafter.  The drafter shares the target's embedding
 * table and LM head ([digest] Method, Training §4.2 step 6; Paper vs code
 * "Embedding and head").  embed, head and fc are borrowed like wo and w_down
 * (in place until dflash_destroy, 16-byte aligned). */
typedef struct {
    const void* embed;                     /* [V, d] */
    const void* head;                      /* [V, d] */
    const float* final_norm;               /* [d] */
    const dflash_layer_weights* target;    /* host array of target_layers entries */
    const void* fc;                        /* W_c [d, k*d] (context fusion, [review] §5.1 eq. 9) */
    const float* fc_norm;                  /* [d] */
    const dflash_layer_weights* draft;     /* host array of draft_layers entries */
    const float* draft_norm;               /* [d] drafter's final RMSNorm */
} dflash_weights;

typedef struct {
    int64_t rounds;            /* draft+verify rounds run by dflash_generate */
    int64_t tokens;            /* tokens emitted, first tokens included */
    int64_t accepted;          /* accepted drafts, summed over sequences and rounds */
    double prefill_ms;         /* device time, CUDA events on the session stream */
    double draft_ms;           /* summed over rounds */
    double verify_ms;          /* summed over rounds */
    int64_t kernel_launches;   /* kernels this session has launched */
} dflash_stats;

typedef struct dflash_ctx dflash_ctx; /* opaque; owned by the library */

/* Create a session: validate cfg, allocate the paged target KV cache and the
 * draft context cache (one pool of kv_pool_tokens / 64 pages of 64 tokens,
 * shared by the batch: a sequence takes pages from the pool as it grows, so
 * a ragged batch needs only the sum of its lengths, and every page returns to
 * the pool at the next prefill), all round buffers for max_batch sequences of
 * up to max_seq_len tokens (nothing is allocated later), and pack the q/k/v
 * and gate/up matrices into the library's layout.  Those packed copies are the session's only weight
 * memory: (H + 2 H_kv) hd d + 2 F d elements per layer, about 13 of the 19.7 GB
 * of a Qwen3-8B-shaped target with its 5-layer drafter; the caller's wq, wk, wv,
 * w_gate and w_up may be freed once this returns, and every other matrix is
 * used in place.  cuda_stream is a cudaStream_t (NULL = legacy default stream).
 * Errors: E_INVAL (cfg, a NULL or misaligned borrowed weight), E_NOMEM, E_CUDA.
 * *out is NULL on failure. */
dflash_status dflash_init(const dflash_config* cfg, const dflash_weights* w, void* cuda_stream,
                          dflash_ctx** out);

/* Target prefill of a new batch ([digest] greedy decoding-round pseudocode,
 * prefill and fuse steps; [review] §5.1): a causal forward over each prompt,
 * the first token = argmax of the last row, and the context feature
 * RMSNorm(W_c [h_l1; ...; h_lk]) of every prompt position injected as keys and
 * values into every draft layer.  Afterwards each sequence's committed length
 * n_i = prompt_lens[i] and its anchor is its first token.
 * prompt_lens: host [batch]; prompt_tokens: host, concatenated (sum of lens);
 * first_tokens: host [batch] output.
 * Errors: E_INVAL (batch outside [1, max_batch], a length < 1, a token outside
 * [0, V)), E_CAPACITY (length + block_size > max_seq_len, or the KV page pool
 * cannot hold every prompt + block_size), E_CUDA. */
dflash_status dflash_prefill(dflash_ctx* ctx, int32_t batch, const int32_t* prompt_lens,
                             const int32_t* prompt_tokens, int32_t* first_tokens);

/* Set the block size B of the following rounds to block_size, between 1 and
 * the configured block size (the drafter's training block).  A drafter trained
 * at one block size still drafts well at a smaller one, and a smaller block
 * is cheaper to verify when the target is compute-bound at large batch
 * ("DFlash" wiki, Ablations: block size; [digest] Pitfalls, on §5.5.4 and tab. 8).
 * Weights, caches and committed lengths are unchanged; a pending context
 * append keeps the block size of the verify that produced it.  The sizes of
 * every round array (draft_tokens [batch, B-1], the sampled calls' uniforms,
 * dflash_inspect's per-row items) follow the new B from the next draft on,
 * and dflash_inspect's kept rows of earlier rounds are read with the current B.
 * Allowed before a prefill and between a verify and the next draft.
 * Errors: E_INVAL (ctx NULL or block_size outside [1, configured B]),
 * E_STATE (a draft awaits its verify). */
dflash_status dflash_set_block_size(dflash_ctx* ctx, int32_t block_size);

/* The block size of the next round (-1 for a NULL ctx). */
int32_t dflash_block_size(const dflash_ctx* ctx);

/* One drafting pass ([digest] Inference steps 2-3 and the draft-layer
 * pseudocode; [review] §5.1 eq. 10).  First appends the context features of
 * the anchor and accepted drafts of the previous verify (a_i + 1 rows per
 * sequence), then runs the drafter once over [anchor, MASK x (B-1)] at
 * positions n_i .. n_i+B-1, with bidirectional attention over
 * [context K/V ; block K/V], and writes the argmax of the shared head on the
 * B-1 mask rows.  The stored context entries are not modified.
 * draft_tokens: [batch, B-1] int32, host or device.
 * Errors: E_STATE (no prefill, or a draft not yet verified), E_CAPACITY, E_CUDA. */
dflash_status dflash_draft_block(dflash_ctx* ctx, int32_t* draft_tokens);

/* Verify a proposal with one causal target pass over [anchor, d_1..d_{B-1}]
 * at positions n_i .. n_i+B-1 ([digest] Inference step 4; [review] §4.1,
 * Algorithm 1).  Accepts the longest prefix with d_j equal to the target's
 * argmax at the position before it (a_i drafts), sets bonus_i to the target's
 * argmax after that prefix, keeps target cache entries for the anchor and the
 * a_i accepted drafts only (n_i += a_i + 1), and makes bonus_i the next
 * anchor.  The proposal need not come from dflash_draft_block: any tokens in
 * [0, V) are verified exactly.
 * draft_tokens: [batch, B-1] int32 input; accepted, bonus: [batch] int32
 * outputs; each host or device.
 * Errors: E_STATE (no dflash_draft_block since the last verify), E_INVAL
 * (host token outside [0, V)), E_DEVICE_CHECK (device token outside [0, V),
 * reported at the next synchronising call), E_CUDA. */
dflash_status dflash_verify(dflash_ctx* ctx, const int32_t* draft_tokens, int32_t* accepted,
                            int32_t* bonus);

/* Temperature sampling (T > 0): speculative rejection sampling ([review] §4.2
 * eq. 6-8 and Algorithm 1 steps 2-3, 7-8 and 10; [digest] Paper vs code
 * "Sampling rule").  The method's random numbers are inputs: every draw is
 * the lowest token z whose cumulative weight exceeds u * total weight, for a
 * caller-supplied uniform u in [0, 1).  Every law, the drafter's and the
 * target's, is filtered by the setting of dflash_set_sampling_filter (off by
 * default).  The vocabulary must fit the sampling kernels (each of up to 8
 * CTAs of a row stages its share of the row in shared memory: about 390K
 * tokens), else E_INVAL.
 *
 * dflash_draft_block_sampled: as dflash_draft_block, then the proposal of
 * mask row j is drawn from q_j = softmax(draft logits_j / T), filtered, with
 * u_draft[s*(B-1) + j-1]; the laws q are kept for the next verify.
 * u_draft: [batch, B-1] float, host (each in [0, 1), else E_INVAL) or device
 * (clamped to [0, 1)); draft_tokens: [batch, B-1] int32 output, host or device.
 * Errors: as dflash_draft_block, plus E_INVAL (T not positive and finite).
 *
 * dflash_verify_sampled: one causal target pass as dflash_verify; with
 * p_j = softmax(verify logits_j / T), filtered, proposal j (block row j+1) is accepted
 * while u_verify[s*B + j] < min(1, p_j(y)/q_{j+1}(y)); at the first rejection
 * the emitted token is drawn from [p_a - q_{a+1}]_+ (normalised), else from
 * p_{B-1}, with u_verify[s*B + B-1].  Caches keep the anchor and the a_i
 * accepted rows (n_i += a_i + 1); the emitted token is the next anchor.
 * u_verify: [batch, B] float (host or device, as above); draft_tokens:
 * [batch, B-1] int32 input (the laws are those of the preceding sampled draft);
 * accepted, emitted: [batch] int32 outputs, host or device.
 * Errors: E_STATE (no dflash_draft_block_sampled since the last verify),
 * E_INVAL (T, NULL, host token or uniform out of range), E_DEVICE_CHECK
 * (device token outside [0, V): treated as a rejection), E_CUDA. */
/* Top-k / top-p filter of the sampled round's laws ([digest] Paper vs code
 * "Sampling rule": they apply to both the draft and the target
 * distributions).  After the temperature, tokens rank by logit, highest
 * first, equal logits in increasing id; top-k keeps the first top_k of them
 * (0: all); top-p then keeps each token whose mass ranked before it, under
 * the top-k law renormalised, is below top_p (1: all); the kept tokens'
 * probabilities are renormalised, and eq. 6-8 apply to the filtered laws.
 * The GPU takes each mass in fp32 and sums them exactly in 2^-32 fixed point
 * (relative to the row's largest probability), so a token whose preceding
 * mass is within about 1e-6 of top_p may fall on either side; the kept set
 * is the same on every run.  Applies from the next
 * sampled draft on; allowed whenever no draft awaits its verify.
 * Errors: E_INVAL (ctx NULL, top_k < 0, top_p outside (0, 1]), E_STATE
 * (between a draft and its verify), E_CUDA. */
dflash_status dflash_set_sampling_filter(dflash_ctx* ctx, int32_t top_k, float top_p);

dflash_status dflash_draft_block_sampled(dflash_ctx* ctx, float temperature, const float* u_draft,
                                        int32_t* draft_tokens);
dflash_status dflash_verify_sampled(dflash_ctx* ctx, float temperature, const int32_t* draft_tokens,
                                    const float* u_verify, int32_t* accepted, int32_t* emitted);

/* The drafter's training forward, loss value only ([review] §6 eq. 12 and
 * Algorithm 2; [digest] Training §4.2).  The target runs once, causally, over
 * the clean sequence tokens[0..n_tokens); for each anchor a the block
 * [tokens[a], MASK x (B-1)] at positions a .. a+B-1 attends to the fused
 * target features of positions < a and to itself; the loss is the mean over
 * anchors of sum_{k=1}^{B-1} exp(-(k-1)/lambda) * -log q_k(tokens[a+k]).
 * All blocks run in one drafter pass: block i uses sequence slot i+1, whose
 * page table shares slot 0's context pages below its anchor's page.
 * tokens: host [n_tokens]; anchors: host [n_anchors], each in [1, n_tokens-B];
 * loss: host float.  Needs B >= 2, n_anchors + 1 <= max_batch and
 * n_tokens + B <= max_seq_len.  Leaves the session empty (prefill before the
 * next round).  Errors: E_INVAL (NULL, anchor range, lambda <= 0, B < 2),
 * E_CAPACITY, E_DEVICE_CHECK, E_CUDA. */
dflash_status dflash_train_forward(dflash_ctx* ctx, int32_t n_tokens, const int32_t* tokens, int32_t n_anchors,
                                   const int32_t* anchors, float lambda, float* loss);

/* Greedy speculative generation ([digest] greedy decoding-round pseudocode):
 * prefill, then rounds of draft_block + verify until every sequence has
 * max_new_tokens tokens (the first token counts); each sequence's output is
 * cut to max_new_tokens.  out_tokens: host [batch, max_new_tokens];
 * out_lens: host [batch] (always max_new_tokens); stats may be NULL. */
dflash_status dflash_generate(dflash_ctx* ctx, int32_t batch, const int32_t* prompt_lens,
                              const int32_t* prompt_tokens, int32_t max_new_tokens, int32_t* out_tokens,
                              int32_t* out_lens, dflash_stats* stats);

/* Inspection of session state (for tests and profiling).  Copies into host
 * memory; synchronises the stream.  *written receives the byte count.
 *   DFLASH_INSPECT_LENGTHS        int32 [batch]: committed length n_i
 *   DFLASH_INSPECT_ANCHORS        int32 [batch]
 *   DFLASH_INSPECT_POSTERIOR      int32 [batch, B]: target argmax of the last verify
 *   DFLASH_INSPECT_TARGET_K/V     dtype [n_seq, H_kv, hd] of (seq, layer), n_seq committed rows
 *   DFLASH_INSPECT_DRAFT_K/V      same for the draft context cache
 *   DFLASH_INSPECT_LOGITS_PREFILL fp32 [batch, V]   (needs DFLASH_FLAG_KEEP_LOGITS)
 *   DFLASH_INSPECT_LOGITS_DRAFT   fp32 [batch, B, V] (all B rows of the last draft)
 *   DFLASH_INSPECT_LOGITS_VERIFY  fp32 [batch, B, V]
 *   DFLASH_INSPECT_STATS          dflash_stats
 *   DFLASH_INSPECT_HIDDEN_VERIFY  fp32 [batch, B, d]: final residual of the last verify
 *   DFLASH_INSPECT_PROFILE        dflash_profile_entry [DFLASH_K_COUNT] accumulated since the last reset
 * Errors: E_INVAL (unknown item, seq/layer out of range, bytes too small). */
enum {
    DFLASH_INSPECT_LENGTHS = 1,
    DFLASH_INSPECT_ANCHORS = 2,
    DFLASH_INSPECT_POSTERIOR = 3,
    DFLASH_INSPECT_TARGET_K = 4,
    DFLASH_INSPECT_TARGET_V = 5,
    DFLASH_INSPECT_DRAFT_K = 6,
    DFLASH_INSPECT_DRAFT_V = 7,
    DFLASH_INSPECT_LOGITS_PREFILL = 8,
    DFLASH_INSPECT_LOGITS_DRAFT = 9,
    DFLASH_INSPECT_LOGITS_VERIFY = 10,
    DFLASH_INSPECT_STATS = 11,
    DFLASH_INSPECT_HIDDEN_VERIFY = 12,
    DFLASH_INSPECT_PROFILE = 13,       /* dflash_profile_entry [DFLASH_K_COUNT]; needs DFLASH_FLAG_PROFILE */
    DFLASH_INSPECT_PROFILE_RESET = 14  /* clears the profile; copies nothing */
};
dflash_status dflash_inspect(dflash_ctx* ctx, int32_t what, int32_t seq, int32_t layer, void* host_dst,
                             size_t bytes, size_t* written);

/* Turn kernel-class timing on (1) or off (0) for this session.  While on,
 * every kernel class launch is bracketed by CUDA events on the session stream
 * and its algorithmic bytes and flops are recorded; read the totals with
 * DFLASH_INSPECT_PROFILE.  Timing adds event records between launches, so
 * headline timings are taken with it off.  Errors: E_INVAL (ctx NULL), E_CUDA. */
dflash_status dflash_set_profiling(dflash_ctx* ctx, int32_t on);

/* Maximum scratch, in bytes, of dflash_head_argmax_noalloc. */
enum { DFLASH_NOALLOC_SCRATCH_BYTES = 16 << 20 };

/* Shared-head argmax for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this call; it exists for deployment.  Some
 * callers cannot call cudaMalloc or any allocator: code running inside
 * another framework's fixed memory pool, an embedded runtime whose allocator
 * is locked, or a process whose device memory budget is settled before this
 * library is loaded.  Such a caller cannot create a session (dflash_init
 * allocates), but can still pick tokens from final hidden states with this
 * call: out[r] = argmax_v ( RMSNorm(x[r]) * norm_w ) . head[v], ties to the
 * lowest id.  It queues three kernels - an RMSNorm of the rows into the
 * element type of head, the head GEMM (tensor cores for bf16), and a row
 * argmax - plus a check of its error word.  dflash_verify computes the same
 * quantity with the norm and the argmax fused into its head GEMM; in bf16 the
 * two can pick different tokens where the two largest logits lie within
 * bf16 rounding of each other.
 *
 * Arguments (all device pointers except cuda_stream):
 *   dtype   DFLASH_DTYPE_F32 or DFLASH_DTYPE_BF16: element type of head
 *   x       fp32 [rows, d_model] hidden states (not modified)
 *   norm_w  fp32 [d_model] RMSNorm scale;  eps: RMSNorm epsilon (> 0)
 *   head    [vocab, d_model] LM head
 *   out     int32 [rows] token ids (written)
 *   cuda_stream  cudaStream_t the kernels are queued on (NULL = legacy default)
 * x, norm_w and head must be 16-byte aligned.  The call queues its kernels and
 * returns without synchronising.
 *
 * Memory: it allocates nothing.  Its intermediates (the normalised rows and
 * the fp32 logits, rows * (d_model * elem + vocab * 4) bytes plus alignment)
 * and a device error word live in one fixed array of
 * DFLASH_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU which loads this
 * library holds until the process exits.  Larger requests are rejected with
 * DFLASH_E_INVAL before anything is queued (for example at vocab 151936 and
 * d_model 4096 in bf16, up to 27 rows fit).
 * The first call on each device looks up that array's device address with
 * the device current; make that first call before any CUDA stream capture.
 * All calls share the array and it keeps the last call's contents; each call
 * clears its error word first, and nothing else needs to start at zero.
 * Calls that overlap on the GPU (on different streams, or from different
 * threads) race on the array: order them.
 * Errors: E_INVAL (NULL or misaligned pointer, bad sizes, request above the
 * maximum), E_CUDA (a launch failed or a kernel could not be prepared); the
 * text is available from dflash_last_error(NULL).  Because the call does not
 * synchronise, a failure on the device is reported in the output instead: if
 * a bounded device-side wait inside the head GEMM ran out (it should never),
 * every out[r] is -1, which is not a token id. */
dflash_status dflash_head_argmax_noalloc(int32_t dtype, const float* x, const float* norm_w, float eps,
                                         const void* head, int32_t rows, int32_t d_model, int32_t vocab,
                                         int32_t* out, void* cuda_stream);

/* Release every library-owned buffer.  NULL is a no-op. */
void dflash_destroy(dflash_ctx* ctx);

/* Text of the last failure on ctx (or of the last failed dflash_init when ctx
 * is NULL).  Valid until the next call on the same ctx. */
const char* dflash_last_error(const dflash_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
