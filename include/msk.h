/*
 * msk.h - C ABI of the persistent MoE verify-step kernel library (libmsk.so).
 *
 * One call of msk_decode_step runs the verify pass of a speculative decode
 * step at batch size one: T (<= 16) tokens through every decoder layer of a
 * sliding-window / global-attention mixture-of-experts transformer, one
 * persistent kernel launch per layer.  Sources, by page title and section:
 *   [newruntime] "Muse Spark Open Ultrafast: Pushing beyond 1,000 Tokens per
 *                second" (newruntime.com), "What happened": 62 decoder
 *                layers (46 sliding-window over the previous 2,048 tokens,
 *                16 global), 8 of 256 experts per token, NVFP4 experts with
 *                some layers in bf16, 16 tokens verified in one pass.
 *   [orcarouter] "Muse Spark Open: 1.109 token al secondo sono un cambiamento
 *                di kernel, non un cambiamento di modello" (orcarouter.ai),
 *                "Dove si colloca il confine del kernel": each launch covers
 *                one layer's attention through the next layer's QKV
 *                projection and KV write; a pooler shrinks each token vector
 *                before the experts and an unpooler restores it; fp4 after
 *                the first expert GEMM, bf16 after the second.
 *   [ai4snews]   "Muse Spark Open decoding passes 1,000 tokens per second..."
 *                (ai4snews.wisdomeyes.cn), "Interpretation": speculative L2
 *                prefetch of the 14 experts the previous step used most.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless a comment says host.
 *   - The caller owns every buffer it passes.  The library copies what it
 *     needs from weights during msk_load_layer (repacking them into its own
 *     device memory); caller weight buffers may be freed after that call.
 *   - Work is enqueued on the given stream.  msk_layer_step and
 *     msk_decode_step synchronise that stream before returning, to read the
 *     device error word; they return MSK_ERR_TIMEOUT if a bounded device
 *     wait ran out (the device context stays usable and the next call
 *     re-initialises the device synchronisation state).  With the
 *     environment variable MSK_VERBOSE_ERRORS set, the device error word
 *     (code, phase, block) is also printed to stderr.
 *   - No C++ exception crosses this boundary.  A model is not thread-safe;
 *     use one model per host thread / stream.
 *   - Requires an sm_103 device (GB300); otherwise MSK_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef MSK_H_
#define MSK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MSK_OK = 0,
  MSK_ERR_INVALID_ARG = 1,      /* null pointer, bad index, inconsistent sizes */
  MSK_ERR_SHAPE = 2,            /* a dimension the kernels do not support */
  MSK_ERR_ALIGNMENT = 3,        /* a pointer or stride not 16-byte aligned */
  MSK_ERR_BAD_SCALE = 4,        /* an E4M3 block scale is NaN or negative */
  MSK_ERR_UNSUPPORTED_DEVICE = 5,
  MSK_ERR_OOM = 6,
  MSK_ERR_CUDA = 7,             /* a CUDA runtime call failed */
  MSK_ERR_TIMEOUT = 8,          /* a device wait exceeded its time budget */
  MSK_ERR_NOT_LOADED = 9        /* a layer's weights were never loaded */
} msk_status;

typedef struct msk_model msk_model; /* opaque, library-owned */

/* Model configuration.  Supported: hidden, pooled and inter multiples of 128;
 * head_dim 64 or 128; n_q_heads a multiple of n_kv_heads with
 * (n_q_heads / n_kv_heads) * verify_tokens <= 64; verify_tokens <= 16;
 * top_k <= 8; n_experts <= 256 (a multiple of 8); pooled, inter <= 2048;
 * hidden <= 4096.
 * Anything else: msk_create returns MSK_ERR_SHAPE. */
typedef struct {
  int32_t n_layers;
  int32_t hidden;          /* D */
  int32_t n_q_heads;       /* Hq */
  int32_t n_kv_heads;      /* Hkv; query head h reads kv head h / (Hq/Hkv) */
  int32_t head_dim;        /* d */
  int32_t pooled;          /* P: pooler output width, expert input width */
  int32_t n_experts;       /* E */
  int32_t top_k;           /* k */
  int32_t inter;           /* I: expert intermediate width */
  int32_t verify_tokens;   /* T */
  int32_t max_seq;         /* KV cache capacity per layer */
  int32_t prefetch_experts; /* experts prefetched into L2 per layer (14) */
  const uint8_t* layer_is_global; /* HOST [n_layers]: 1 global, 0 sliding */
  int32_t window;          /* sliding window W: keys [p - W + 1, p] */
  float rms_eps;           /* RMSNorm epsilon (1e-6) */
  float rope_theta;        /* RoPE base (1e6) */
  uint64_t wait_budget_ns; /* bound on every device-side wait; 0 = 200 ms */
} msk_model_config;

/* A bf16 matrix [rows][cols], row-major; ld_elems = elements between rows
 * (>= cols, a multiple of 8; 0 means cols). */
typedef struct {
  const void* data;
  int64_t rows, cols, ld_elems;
} msk_bf16_desc;

/* An NVFP4 matrix [rows][cols] (cols a multiple of 128):
 *   packed: [rows][cols/2] bytes, element 2i in the low nibble of byte i,
 *           element 2i+1 in the high nibble; E2M1 codes (bit 3 = sign);
 *   scales: [rows][cols/16] E4M3 codes, one per 16 consecutive elements
 *           along a row (sign bit must be 0, NaN codes are rejected);
 *   tensor_scale: fp32 multiplier of the whole matrix.
 * Value w[r][c] = fp32(e2m1 * e4m3) * tensor_scale. */
typedef struct {
  const uint8_t* packed;
  const uint8_t* scales;
  float tensor_scale;
  int64_t rows, cols;
} msk_nvfp4_desc;

/* One layer's weights.  Dense weights are [out][in] (K-major).
 *   attn_norm, moe_norm : [1][hidden] RMSNorm gains;
 *   w_qkv   : [(Hq + 2 Hkv) d][hidden], rows [q heads | k heads | v heads];
 *   w_o     : [hidden][Hq d];  w_pool : [pooled][hidden];
 *   w_router: [n_experts][pooled];  router_bias : fp32 [n_experts];
 *   w_unpool: [hidden][pooled];
 *   w_gate, w_up : HOST arrays [n_experts] of [inter][pooled] NVFP4;
 *   w_down  : HOST array [n_experts] of [pooled][inter] NVFP4. */
typedef struct {
  msk_bf16_desc attn_norm, moe_norm, w_qkv, w_o, w_pool, w_unpool, w_router;
  const float* router_bias;
  const msk_nvfp4_desc* w_gate;
  const msk_nvfp4_desc* w_up;
  const msk_nvfp4_desc* w_down;
} msk_layer_weights;

/* Creates a model: validates the configuration, checks the device, and
 * allocates the library's scratch (activations between phases, attention
 * partials, synchronisation words).  *out is NULL on failure. */
msk_status msk_create(const msk_model_config* cfg, msk_model** out);

/* Copies layer `layer`'s weights into the library's tiled layouts on the
 * device: dense rows in mma-fragment order, expert codes and block scales
 * interleaved per 16-row unit.  Validates shapes, 16-byte alignment and every
 * E4M3 block scale (MSK_ERR_BAD_SCALE).  Synchronises `stream`.  Loading a
 * layer again replaces it. */
msk_status msk_load_layer(msk_model* m, int32_t layer, const msk_layer_weights* w,
                          void* stream /* cudaStream_t */);

/* Runs ONE persistent launch: attention(layer) .. MoE(layer) .. and, unless
 * `layer` is the last, QKV(layer + 1) with its KV write.
 *   hidden     : [T][hidden] bf16, in: the layer input h; out: h2.
 *   kv_cache   : [n_layers][2 (K, V)][n_kv_heads][max_seq][head_dim] bf16;
 *                K is stored after RoPE.  Rows at the verify positions of
 *                layer `layer` must already be written (by the previous
 *                launch, or by run_prologue on this one).
 *   positions  : HOST [T], positions[t] == positions[0] + t, the last one
 *                < max_seq.  The cached length is positions[0].
 *   prev_routing: [T][top_k] int32 experts this layer chose in the previous
 *                step, or NULL (no speculative prefetch).  Only moves data
 *                into L2: results never depend on it.
 *   routing_out: [T][top_k] int32, or NULL.  Rank order: logit descending,
 *                index ascending on ties.
 *   run_prologue: nonzero = first compute layer `layer`'s own QKV and KV
 *                write from `hidden` (what the previous launch would have
 *                done).
 * The query vectors of the next layer are kept inside the model between
 * calls.  Returns after the stream has completed the launch. */
msk_status msk_layer_step(msk_model* m, int32_t layer, void* hidden, void* kv_cache,
                          const int32_t* positions, const int32_t* prev_routing,
                          int32_t* routing_out, int32_t run_prologue, void* stream);

/* The whole verify step: the prologue of layer 0, then one launch per layer.
 *   prev_routing: [n_layers][T][top_k] int32 or NULL; routing_out:
 *   [n_layers][T][top_k] int32 or NULL.  hidden holds the last layer's h2
 *   (no final norm) on return; the KV rows of every layer are written at
 *   the verify positions. */
msk_status msk_decode_step(msk_model* m, void* hidden, void* kv_cache, const int32_t* positions,
                           const int32_t* prev_routing, int32_t* routing_out, void* stream);

/* The same two calls for a TREE of candidate tokens instead of a chain
 * ([orcarouter] on the draft: the verified block is a tree of candidates
 * generated by the draft model, not a linear chain).
 *   cache_len : S, the number of cached tokens (every position < S holds a
 *               K/V row); S + T <= max_seq.
 *   parents   : HOST [T]; parents[t] is the verify slot of t's parent, an
 *               earlier slot (0 <= parents[t] < t), or -1 for a child of the
 *               last cached token.  parents[t] == t - 1 for every t is the
 *               chain, i.e. msk_layer_step / msk_decode_step with
 *               positions S + t.
 * Slot t has position S + depth(t) (depth = number of verify ancestors),
 * which sets its RoPE angle and its sliding window; its K/V rows are
 * written at cache row S + t (slot order, so that the caller can compact
 * the accepted path afterwards); it attends to the cached keys inside its
 * window and to the verify rows of its ancestors and itself (those whose
 * positions fall inside its window).  MSK_ERR_INVALID_ARG for a parent out
 * of range or S out of range. */
msk_status msk_layer_step_tree(msk_model* m, int32_t layer, void* hidden, void* kv_cache, int32_t cache_len,
                               const int32_t* parents, const int32_t* prev_routing, int32_t* routing_out,
                               int32_t run_prologue, void* stream);
msk_status msk_decode_step_tree(msk_model* m, void* hidden, void* kv_cache, int32_t cache_len,
                                const int32_t* parents, const int32_t* prev_routing, int32_t* routing_out,
                                void* stream);

/* The whole step as one CUDA graph.  The pages run the draft, the verify
 * and the accept of a decode step as one CUDA graph with 97 launches
 * ([newruntime] "What happened"; the plugin's README in [orcarouter]); this
 * is the verify part.
 * msk_step_graph_capture records the n_layers launches of a step (as
 * msk_decode_step would enqueue them) into a graph owned by the model, on a
 * stream of the library's own; nothing runs.  The buffers given here are
 * baked into the graph: every replay reads and writes these same `hidden`,
 * `kv_cache`, `prev_routing` ([n_layers][T][top_k] or NULL) and
 * `routing_out` ([n_layers][T][top_k] or NULL).  Capturing again replaces
 * the graph.  Must not be called while another capture is active on the
 * calling thread.
 * msk_step_graph_launch replays it for one step on `stream`: the cached
 * length `cache_len` and the candidate tree `parents` (HOST [T], as in
 * msk_decode_step_tree; NULL = the chain) are copied to a small device
 * record that every launch reads at its start, so one graph serves every
 * step.  Results are bit-identical to msk_decode_step_tree /
 * msk_decode_step with the same inputs.  Synchronises `stream`; returns
 * MSK_ERR_NOT_LOADED if nothing was captured, MSK_ERR_INVALID_ARG for a bad
 * cache_len or tree.  Launch timing and the phase timeline are not recorded
 * for replays. */
msk_status msk_step_graph_capture(msk_model* m, void* hidden, void* kv_cache, const int32_t* prev_routing,
                                  int32_t* routing_out);
msk_status msk_step_graph_launch(msk_model* m, int32_t cache_len, const int32_t* parents, void* stream);

/* Per-phase device timestamps (%globaltimer, ns) of the most recent call,
 * recorded only while timing is enabled (msk_set_timing).  Layout:
 * [launches][ctas][MSK_TIMELINE_SLOTS], launches in the call's order (one
 * launch, of the layer given, after msk_layer_step); *n receives the number
 * of uint64 written (at most cap). */
#define MSK_TIMELINE_SLOTS 64
msk_status msk_set_timing(msk_model* m, int32_t enable);
msk_status msk_get_timeline(msk_model* m, uint64_t* host_out, size_t cap, size_t* n,
                            int32_t* n_launches, int32_t* n_ctas);

/* Per-launch device durations.  While enabled, msk_layer_step and
 * msk_decode_step record a CUDA event pair on the call's stream around
 * every layer launch; msk_get_launch_ms returns the durations (ms) of the
 * most recent call's launches, in launch order (*n = number written). */
msk_status msk_set_launch_timing(msk_model* m, int32_t enable);
msk_status msk_get_launch_ms(msk_model* m, float* host_out, int32_t cap, int32_t* n);

/* Test hooks (not needed in production).
 * msk_set_wait_budget: device wait bound in ns (0 restores the default).
 * msk_set_fault_injection: CTA `cta` skips its arrival at grid barrier number
 *   `barrier` (counted from 1 within a launch) of every launch; -1 disables.
 *   Used to check that a missing producer ends in MSK_ERR_TIMEOUT. */
msk_status msk_set_wait_budget(msk_model* m, uint64_t ns);
msk_status msk_set_fault_injection(msk_model* m, int32_t barrier, int32_t cta);

/* Copies an intermediate of the most recent launch (device to device) for
 * tests: 0 q stash [T][Hq][d] bf16, 1 attention output [T][Hq d] bf16,
 * 2 h1 [T][D] bf16, 3 pooled [T][P] bf16, 4 router logits [T][E] fp32,
 * 5 fp4 intermediate codes [T k][I/2] (E2M1, element 2i in the low nibble
 * of byte i), 6 its E4M3 scales [T k][I/16],
 * 7 expert outputs [T k][P] bf16 (slot t*k + r), 8 combined expert output
 * [T][P] bf16, 9 the experts ranked for the speculative L2 prefetch [33]
 * int32 (count n, then n expert ids, most used in prev_routing first).  Copies min(bytes, size of the buffer); *copied = that. */
msk_status msk_debug_scratch(msk_model* m, int32_t which, void* dst, size_t bytes, size_t* copied,
                             void* stream);

/* Dequantises expert `expert`'s matrix `which` (0 gate, 1 up, 2 down) of a
 * loaded layer by reading the library's repacked layout, into out
 * ([rows][cols] fp32, device).  Bit-exact with fp32(e2m1*e4m3)*tensor_scale. */
msk_status msk_debug_dequant(msk_model* m, int32_t layer, int32_t expert, int32_t which,
                             float* out, void* stream);

/* Test hook: the E2M1 code (round-to-nearest-even, saturating; sign bit
 * kept for negative values that round to zero) and the E4M3 code (same rules)
 * of each of the n DEVICE floats in x, written to the DEVICE byte arrays e2m1
 * and e4m3, through the very conversion routines the kernels use for the
 * activation quantiser.  Synchronises `stream`. */
msk_status msk_debug_convert(const float* x, int64_t n, uint8_t* e2m1, uint8_t* e4m3, void* stream);

/* Runs the kernel's activation quantiser on x ([rows][cols] fp32, cols a
 * multiple of 16, device): writes E2M1 codes (one per byte) to codes
 * [rows][cols] and E4M3 scales to scales [rows][cols/16].  Standalone (no
 * model). */
msk_status msk_debug_quantize(const float* x, int64_t rows, int64_t cols, uint8_t* codes,
                              uint8_t* scales, void* stream);

/* Test hook: one block-scaled NVFP4 tile on the tensor cores (tcgen05
 * kind::mxf4nvf4, the instruction the expert GEMMs use), through the same
 * shared-memory operand layouts and scale-factor placement as the layer
 * kernel:  d[128][16] = A[128][K] * B[b_rows][K]^T in fp32, rows of B past
 * b_rows taken as zero.
 *   a_codes : [128][K/2] E2M1 codes, element 2i in the low nibble of byte i;
 *   a_scales: [128][K/16] E4M3 block scales (one per 16 elements of K);
 *   b_codes, b_scales: the same for B's b_rows (1..16) rows;
 *   K: 128..2048, a multiple of 128; d: [128][16] fp32.  All DEVICE.
 * Value of an element: e2m1 * e4m3 (no tensor scale).  Allocates a 4-byte
 * error word; synchronises `stream`. */
msk_status msk_debug_fp4_gemm(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* b_codes,
                              const uint8_t* b_scales, int32_t b_rows, int32_t K, float* d, void* stream);

/* Split-KV GQA attention of one layer (the layer kernel's attention stage)
 * as a standalone call that allocates no device memory.  The pages describe
 * no such call: it is here for callers that cannot allocate when they need
 * attention, e.g. code drawing all device memory from a serving framework's
 * pre-sized pool, or code that must not allocate while work is being
 * recorded for later replay.
 *   q        : [tokens][n_q_heads][head_dim] bf16, rotated queries;
 *   kv_layer : [2 (K, V)][n_kv_heads][max_seq][head_dim] bf16, one layer's
 *              cache, keys after RoPE, rows up to pos0 + tokens - 1 written;
 *   window   : 0 for global attention, else keys [p - window + 1, p];
 *   out      : [tokens][n_q_heads * head_dim] bf16.
 * Token t sits at position pos0 + t and sees keys up to its own position.
 * Supported: head_dim 64 or 128, tokens <= 16, (n_q_heads / n_kv_heads) *
 * tokens <= 64, n_q_heads * head_dim <= 4096, n_kv_heads <= the device's SM
 * count (each kv head needs at least one block); else MSK_ERR_SHAPE.
 * Scratch (per-block partial results and synchronisation words) lives in
 * one fixed 6 MiB array inside the library on every GPU that loads it, kept
 * until the process exits; a call whose shape needs more (SM count * 64 *
 * (head_dim + 2) * 4 bytes + 512) returns MSK_ERR_SHAPE.  The first call on
 * a device looks up that array's device address and sets the kernels'
 * shared-memory limit (guarded by a mutex, so first calls from several host
 * threads are safe).  All calls share the array: calls that overlap on the
 * GPU race, so serialise them.  The synchronisation words are cleared at the
 * start of every call.  The call synchronises `stream` before returning (to
 * read the device error word: MSK_ERR_TIMEOUT if a device wait ran out), so
 * it cannot run while `stream` is being captured into a CUDA graph. */
msk_status msk_attention_noalloc(const void* q, const void* kv_layer, int32_t tokens, int32_t n_q_heads,
                                 int32_t n_kv_heads, int32_t head_dim, int32_t max_seq, int32_t pos0,
                                 int32_t window, void* out, void* stream);

/* Number of SMs (= CTAs per launch) the model uses, and bytes of device
 * memory it owns. */
msk_status msk_get_info(msk_model* m, int32_t* n_ctas, int64_t* device_bytes);

const char* msk_status_string(msk_status s);
void msk_destroy(msk_model* m);

#ifdef __cplusplus
}
#endif
#endif /* MSK_H_ */
