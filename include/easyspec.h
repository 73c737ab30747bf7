/*
 * easyspec.h -- C ABI of libeasyspec.so: EasySpec layer-parallel ("fuzzy")
 * speculative decoding on one NVIDIA B300 (sm_103a).
 *
 * Method sources (web pages describing the method):
 *   [ABS]  "EasySpec: Layer-Parallel Speculative Decoding for Efficient
 *          Multi-GPU Utilization", arXiv abstract (index card page, 2502.02493).
 *   [DISC] The same paper's OpenReview discussion page (paperhub.cn): author
 *          replies on Table 4 / Appendix B.1 (layer sets), Figure 1(b) /
 *          Table 4 (attention-only parallelism), Figure 2 (fuzzy KV and its
 *          replacement) and Table 3 (normalised hidden states).
 *   [SD]   The speculative-sampling rule of the works [ABS] builds on:
 *          Leviathan et al., "Fast Inference from Transformers via
 *          Speculative Decoding"; Chen et al., "Accelerating Large Language
 *          Model Decoding with Speculative Sampling".
 *
 * Conventions for every entry point
 *   - No C++ exception crosses this boundary.  Every call returns an
 *     es_status; on failure a message is kept in the context and returned by
 *     easyspec_last_error().  After ES_ERR_CUDA or ES_ERR_TIMEOUT the context
 *     is poisoned: every later call except easyspec_last_error() and
 *     easyspec_destroy() returns ES_ERR_STATE.
 *   - "device" pointers are CUDA device addresses on the current device;
 *     "host" pointers are ordinary CPU memory (pageable or pinned).
 *   - Weights are BORROWED: the caller allocates them (e.g. with PyTorch),
 *     keeps them alive and unchanged until easyspec_destroy().  The KV caches,
 *     activations and probability buffers are OWNED by the context and freed
 *     by easyspec_destroy().
 *   - All work is issued on the stream given in es_config (0 = the legacy
 *     default stream).  Calls that return host results synchronise that
 *     stream before returning; the others are asynchronous.
 *   - Matrices are row-major [out_features, in_features].  Every in_features
 *     (d, ffn, n_heads*head_dim) must be a multiple of 8, head_dim a multiple
 *     of 8 and <= 256, and n_heads a multiple of n_kv_heads with at most 16
 *     query heads per kv head (ES_ERR_ARG).
 */
#ifndef EASYSPEC_H_
#define EASYSPEC_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ES_API __attribute__((visibility("default")))
#else
#define ES_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ES_OK = 0,
    ES_ERR_ARG = -1,      /* invalid argument or shape                         */
    ES_ERR_OOM = -2,      /* device allocation failed                          */
    ES_ERR_CUDA = -3,     /* a CUDA call failed (context poisoned)             */
    ES_ERR_TIMEOUT = -4,  /* a bounded device-side wait gave up (poisoned)     */
    ES_ERR_STATE = -5,    /* call out of order, or context poisoned            */
    ES_ERR_CAPACITY = -6  /* a sequence would exceed max_seq                   */
} es_status;

enum { ES_DTYPE_F32 = 0, ES_DTYPE_BF16 = 1 };

/* [DISC] Figure 1(b)/Table 4 reply: only attention runs layer-parallel and
 * the MLPs stay sequential (ES_ATTN_ONLY).  ES_FULL_LAYER: attention and MLP
 * of every layer of a set read the set input and all their residual deltas
 * are summed onto it, so the set's QKV and gate/up projections form one wide
 * pass over the shared input and its o/down projections one K-concatenated
 * pass producing the summed delta.  A set of one layer is the exact layer in
 * both modes. */
enum { ES_ATTN_ONLY = 0, ES_FULL_LAYER = 1 };

/* Llama-style decoder shape: RMSNorm (eps), rotary embedding (rope_theta,
 * element i paired with i + head_dim/2), grouped-query attention, SwiGLU MLP,
 * untied output head.  dtype applies to weights and KV cache; activations and
 * accumulation are float32. */
typedef struct {
    int n_layers, d, n_heads, n_kv_heads, head_dim, ffn, vocab;
    float rope_theta, eps;
    int dtype; /* ES_DTYPE_* */
} es_model_shape;

/* Device pointers, borrowed.  Per-layer arrays are HOST arrays of n_layers
 * device pointers.  Shapes: embed, lm_head [vocab, d]; final_norm, attn_norm,
 * mlp_norm [d]; wq [n_heads*head_dim, d]; wk, wv [n_kv_heads*head_dim, d];
 * wo [d, n_heads*head_dim]; wgate, wup [ffn, d]; wdown [d, ffn].
 * Every pointer must be 16-byte aligned. */
typedef struct {
    const void *embed, *lm_head, *final_norm;
    const void *const *attn_norm, *const *wq, *const *wk, *const *wv, *const *wo;
    const void *const *mlp_norm, *const *wgate, *const *wup, *const *wdown;
} es_weights;

typedef struct {
    es_model_shape draft, base;
    int max_batch;            /* sequences decoded together, 1..64            */
    int max_seq;              /* KV capacity per sequence (tokens)            */
    int max_gamma;            /* largest gamma accepted by draft_step, 1..16  */
    int parallel_mode;        /* ES_ATTN_ONLY or ES_FULL_LAYER                */
    /* Explicit layer sets ([DISC] Table 4 reply: "a change in configuration
     * is enough"): n_groups start indices, increasing, group_starts[0] == 0.
     * NULL: sets come from the k passed to draft_step, by the rule of [DISC]
     * (Table 4 / Appendix B.1 reply): layer 0 and layer L-1 alone, layers
     * 1..L-2 in aligned blocks [mk, mk+k-1]. */
    const int *group_starts;
    int n_groups;
    void *cuda_stream;        /* cudaStream_t, or NULL for the default stream */
} es_config;


/* Per-run counters filled by generate() (may be NULL). */
typedef struct {
    int64_t phases;           /* drafting-and-verification iterations run     */
    int64_t drafted;          /* draft tokens proposed to unfinished sequences */
    int64_t accepted;         /* of those, accepted                           */
    int64_t emitted;          /* tokens committed (before cutting to max_new) */
    int64_t kernel_launches;  /* kernels of this library launched while decoding */
    double prefill_ms, decode_ms;  /* host wall-clock                          */
} es_stats;

typedef struct es_ctx es_ctx;

/* Create a context: validates shapes (draft.vocab == base.vocab: draft and
 * base must share token ids, [DISC] reply on cross-family drafting), binds the
 * borrowed weights, allocates the paged KV caches (64-token pages) and the
 * workspace on the device current at the call.  *out is NULL on failure. */
ES_API es_status easyspec_init(const es_config *cfg, const es_weights *draft,
                        const es_weights *base, es_ctx **out);

/* Load B prompts (host int32 [B, P], P >= 1) and run the exact prefills:
 * the base over x_0..x_{P-2} and the draft over the same tokens, leaving the
 * last prompt token pending in both.  Resets the phase counter. */
ES_API es_status easyspec_prefill(es_ctx *ctx, const int32_t *prompts, int B, int P);

/* Bonus calibration ([ABS]; [DISC] Figure 2 reply): one exact draft forward
 * over the last gamma+1 committed tokens of every sequence, which covers all
 * tokens committed since the last calibration; it overwrites their fuzzy KV
 * entries with exact ones and yields q_1, from which d_1 is drawn (slot 0 of
 * the phase's draws).  Runs implicitly in draft_step when still pending.
 * gamma as in draft_step; temperature 0 = greedy. */
ES_API es_status calibrate_kv(es_ctx *ctx, int gamma, float temperature, uint64_t seed);

/* Calibration ablation ([ABS]; [DISC] first reply: without calibration the
 * fuzzy errors accumulate).  on = 1 (the default after easyspec_init) runs
 * the calibration above.  on = 0 keeps, after each verify_step, the
 * layer-parallel KV entries of the accepted drafts d_1..d_min(a, gamma-1);
 * the exact draft forward that starts the next phase then covers only the
 * committed positions that hold no draft entry (the bonus token, and d_gamma
 * when every draft was accepted) and still yields q_1.  Takes effect at the
 * next calibrate_kv / draft_step / es_decode / generate; the positions kept
 * so far stay as they are.  ES_ERR_ARG unless on is 0 or 1; ES_ERR_STATE
 * between a draft_step (or calibrate_kv) and its verify_step. */
ES_API es_status es_set_calibration(es_ctx *ctx, int on);

/* Drafting ([ABS]; [DISC] Table 4 and Figure 2 replies): calibration (if
 * pending) then gamma-1 layer-parallel draft forwards of d_1..d_{gamma-1}
 * under layer-set size k (ignored, and must be 0, when explicit sets were
 * configured), each writing fuzzy KV entries and drawing the next draft
 * token.  draft_out: host int32 [B, gamma] or NULL. */
ES_API es_status draft_step(es_ctx *ctx, int k, int gamma, float temperature,
                     uint64_t seed, int32_t *draft_out);

/* Verification and acceptance ([ABS]; [SD]): one exact base forward over
 * [x_{n-1}, d_1..d_gamma] per sequence giving p_1..p_{gamma+1}, then the
 * accept test u*q_i(d_i) < p_i(d_i) (float32, u from slot gamma+i-1) and the
 * residual / bonus draw (slot 2*gamma); greedy (temperature 0) compares
 * argmaxes.  Commits n_accepted+1 tokens per sequence and truncates both
 * caches.  Must follow draft_step with the same gamma, temperature and seed.
 * n_accepted: host int32 [B] or NULL; tokens_out: host int32 [B, gamma+1]
 * or NULL (entries past n_accepted+1 are -1). */
ES_API es_status verify_step(es_ctx *ctx, float temperature, uint64_t seed,
                      int32_t *n_accepted, int32_t *tokens_out);

/* Whole speculative generation ([ABS]: draft with layer-parallel sets, verify
 * the drafts in one base forward, calibrate the draft KV; [DISC] Figure 2
 * reply: fuzzy entries live for one phase and are then replaced): prefill,
 * then phases of draft_step + verify_step until every sequence has max_new new tokens (a sequence that
 * has them stops committing while the others finish).  out: host int32
 * [B, max_new].  Needs P + max_new + 2*gamma + 2 <= max_seq
 * (ES_ERR_CAPACITY). */
ES_API es_status generate(es_ctx *ctx, const int32_t *prompts, int B, int P,
                   int max_new, int gamma, int k, float temperature,
                   uint64_t seed, int32_t *out, es_stats *stats);

/* The decoding loop of generate() ([ABS]; [DISC] Figure 2 reply) without
 * the prefill.  Decode max_new more tokens for every loaded sequence (after
 * easyspec_prefill or a previous decode): phases of draft_step + verify_step
 * as in generate(), with the tokens left on the device (read them with
 * es_read_tokens).  Needs n + max_new + 2*gamma + 2 <= max_seq for every
 * sequence of current length n (ES_ERR_CAPACITY). */
ES_API es_status es_decode(es_ctx *ctx, int max_new, int gamma, int k, float temperature,
                           uint64_t seed, es_stats *stats);

/* Timing for measurement.  on = 1 (per kernel): every later launch runs
 * outside CUDA graphs, bracketed by CUDA events on the context's stream, and
 * is reported under "<model>.<step>" labels.  on = 2 (per phase part): the
 * CUDA graphs stay; each graph launch is bracketed by events ("phase.draft",
 * "phase.verify", "phase.calibrate", "phase.fuzzy"; es_decode then launches
 * calibration and the fuzzy drafts as two graphs).  on = 0: off.
 * es_profile_read() reports, per label (entries idx = 0, 1, ... until
 * ES_ERR_ARG), the summed event time in ms, the launch count and the
 * algorithmic bytes of those launches (weights plus activations moved; 0 for
 * kernels whose traffic is not modelled and for parts).  es_profile() resets
 * the totals; another `on` is ES_ERR_ARG. */
ES_API es_status es_profile(es_ctx *ctx, int on);
ES_API es_status es_profile_read(es_ctx *ctx, int idx, char *name, int name_cap, double *ms,
                                 int64_t *launches, double *bytes);

/* Accept/resample alone ([SD]) on caller data, for checking.  Device
 * pointers: p float32 [B, gamma+1, V] (greedy: logits), q float32
 * [B, gamma, V] (greedy: logits), d int32 [B, gamma], u uint64 [B, gamma+1]
 * (gamma accept draws, then the residual/bonus draw); outputs n_acc int32 [B]
 * and tok int32 [B, gamma+1] (-1 past n_acc+1).  Synchronous on `stream`. */
ES_API es_status es_accept_resample(const float *p, const float *q, const int32_t *d,
                             const uint64_t *u, int B, int gamma, int V,
                             int greedy, int32_t *n_acc, int32_t *tok,
                             void *stream);

/* es_accept_resample without any device allocation.  The pages have no
 * counterpart.  es_accept_resample allocates its scratch (per-chunk partials,
 * masses, arrival counters) with cudaMalloc on every call; some callers
 * cannot do that where they call: a serving host that reserved the device's
 * memory for its own pool allocator up front (cudaMalloc then fails, or
 * takes memory the pool counts on), and a decode loop that cannot take
 * cudaFree's device-wide synchronisation between tokens.  This entry point
 * works in a fixed array inside the library instead.
 *   Limits: B <= 16, gamma <= 16, and at most 160 vocabulary chunks.  A
 *   chunk is max(512, ceil(V / SMs)) entries, so the call uses
 *   min(SMs, ceil(V / 512)) chunks: any V fits on a device with at most 160
 *   SMs (148 on a B300), and a device with more SMs refuses large V.
 *   Larger sizes return ES_ERR_ARG (with a message on stderr).
 *   The array (about 390 KB) is held by every GPU that loads the library
 *   until the process exits.  It is shared by every call in the process on a
 *   device and keeps the last call's contents (the arrival counters are
 *   cleared at each call): calls that overlap on the GPU -- on different
 *   streams, or from several host threads -- race and must not be issued.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture
 *   begins.
 * Arguments, layouts and results as es_accept_resample; synchronous on
 * `stream`. */
ES_API es_status es_accept_resample_noalloc(const float *p, const float *q, const int32_t *d,
                                            const uint64_t *u, int B, int gamma, int V, int greedy,
                                            int32_t *n_acc, int32_t *tok, void *stream);

/* Integer-quantised categorical draw alone ([SD] sampling step, quantised
 * as the oracle does): for each of B rows of unnormalised float32 weights
 * w [B, V] (device) and one draw u [B] (device), writes the index to
 * idx [B] (device), or -1 when all weights quantise to zero. */
ES_API es_status es_sample(const float *w, const uint64_t *u, int B, int V,
                    int32_t *idx, void *stream);

/* The bounded device-side wait of the tensor-core weight passes on its own
 * (no counterpart in the pages: it checks the library's failure path without
 * a GPU fault).  Those passes wait on mbarriers for their TMA copies and
 * MMAs; every wait gives up after a time limit, sets a device flag and lets
 * the kernel free its tensor memory and return, and the host then reports
 * ES_ERR_TIMEOUT and poisons the context.  This call runs one such wait:
 * thread 0 waits at most limit_ns (1 ns .. 2 s) on a barrier that a second
 * thread arrives at after arrive_ns (< 0: never; at most 1 s).  Returns
 * ES_ERR_TIMEOUT when the wait gave up, ES_OK when the arrival came first,
 * ES_ERR_ARG for limits out of range.  Needs no context; synchronous on
 * `stream`; allocates and frees one int of device memory. */
ES_API es_status es_wait_selftest(int64_t limit_ns, int64_t arrive_ns, void *stream);

/* Copy cached K and V of one layer and sequence, positions [0, n), to host
 * float32 arrays k_out, v_out [n, n_kv_heads, head_dim].  which: 0 draft,
 * 1 base. */
ES_API es_status es_read_kv(es_ctx *ctx, int which, int layer, int seq, int n,
                     float *k_out, float *v_out);

/* Copy the last phase's distributions to host float32:  which 0: draft q
 * [B, gamma, V]; 1: base p [B, gamma+1, V]; 2: draft logits [B, gamma, V];
 * 3: base logits [B, gamma+1, V].  (Greedy phases store logits in q/p.) */
ES_API es_status es_read_dist(es_ctx *ctx, int which, float *out);

/* Copy committed tokens of sequence `seq` to host int32 out[0..n) and return
 * their count in *n_committed (out may be NULL to query the count). */
ES_API es_status es_read_tokens(es_ctx *ctx, int seq, int32_t *out, int cap,
                         int *n_committed);

/* The draft layer sets that set size k gives when no explicit sets are
 * configured ([DISC] reply on Table 4 / Appendix B.1): layer 0 and layer
 * n_layers-1 alone, the layers between in blocks aligned to multiples of k;
 * k = 1 gives one set per layer.  Writes the first layer of each set to
 * starts[0..min(cap, *n_sets)) (host int32, caller-owned) and the number of
 * sets to *n_sets (cap 0 and starts NULL query the count).  Host only: needs
 * no context and no GPU.  ES_ERR_ARG unless n_layers >= 1 and 1 <= k <= 8. */
ES_API es_status es_layer_sets(int n_layers, int k, int32_t *starts, int cap, int *n_sets);

ES_API const char *easyspec_last_error(const es_ctx *ctx);
ES_API void easyspec_destroy(es_ctx *ctx);

#ifdef __cplusplus
}
#endif
#endif /* EASYSPEC_H_ */
