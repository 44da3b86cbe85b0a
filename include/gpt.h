/*
 * gpt.h - C ABI of the GB300 (sm_103a) GPT forward + next-token cross-entropy library.
 *
 * What the library computes (the definitions it follows, by page and section):
 *   x0[b,t]  = E[ids[b,t]] + P[t]                 "第 25 章 从小 GPT 到 GPT-2" §25.1;
 *                                                "预训练一个 Mini GPT（1.24 亿参数）" 第1步
 *   L blocks, pre-norm:  x += attn(LN1 x); x += mlp(LN2 x)              §25.1, 第4步
 *            post-norm:  n = LN1(x + attn x); x = LN2(n + mlp n)        "GPT-1 学习笔记" §3.1-3.2
 *   attn: qkv = a W_attn^T + b (C -> 3C), split into Q, K, U and H heads of D = C/H,
 *         y = softmax(Q K^T / sqrt(D) + M) U with M = -inf for s > t, heads merged,
 *         then c_proj (C -> C)                                          §25.2
 *   mlp:  C -> ffn -> C with GELU (tanh form by default)                §25.3; "GPT-1 学习笔记" §3.6
 *   LN:   (x - mean) / sqrt(var + eps) * g + b, biased variance         第4步; "GPT-1 学习笔记" §3.2
 *   head: logits = h E^T, tied to the token table, no bias              §25.4
 *   loss: mean over all B*T positions of -log softmax(logits)[target]   §25.7; 第6步
 *
 * Conventions
 *   - Every function returns an int status (GPT_OK = 0, else a GPT_E* code);
 *     nothing is thrown across the ABI. gpt_strerror() names a code.
 *   - Weight matrices use the nn.Linear orientation [out, in] (row-major).
 *     A source that stores Conv1D weights [in, out] must transpose exactly
 *     the four projection matrices (§25.5); tables, LayerNorms and biases
 *     are not transposed.
 *   - Device pointers are CUDA device memory of the current device; host
 *     pointers are ordinary (pageable or pinned) host memory.
 *   - Streams are cudaStream_t values passed as void* (NULL = legacy default stream).
 */
#ifndef GPT_GB300_H
#define GPT_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  GPT_OK = 0,
  GPT_EINVAL = 1,      /* null pointer, B or T < 1, B*T > max_tokens, a dimension not a multiple of 8 */
  GPT_ECONFIG = 2,     /* C not divisible by H ("Day 16 从零组装 MiniGPT" §三十八), unsupported head width or C */
  GPT_ESEQ = 3,        /* T > ctx: the position table has no row for it ("Day 16 从零组装 MiniGPT" §三十九) */
  GPT_ETOKEN = 4,      /* a token id or a target outside [0, V); found on the device */
  GPT_ECUDA = 5,       /* a CUDA runtime or driver call failed */
  GPT_ENOMEM = 6,      /* device or pinned-host allocation failed */
  GPT_EDEVICE = 7,     /* a kernel's bounded wait expired or its shared memory was misaligned */
  GPT_EUNSUPPORTED = 8 /* the device is not sm_103 (GB300) or lacks the resources */
};

/* Model hyper-parameters ("Day 16 从零组装 MiniGPT" §三, GPTConfig). */
typedef struct gpt_config {
  int32_t V;           /* vocabulary size */
  int32_t C;           /* hidden width; multiple of 8 */
  int32_t H;           /* attention heads; C % H == 0; D = C/H in {32, 64} on the bf16 path */
  int32_t L;           /* blocks, >= 0 */
  int32_t ctx;         /* rows of the position table = longest sequence */
  int32_t ffn;         /* MLP hidden width (4C in GPT-2); multiple of 8 */
  int32_t norm_mode;   /* 0 pre-norm (GPT-2), 1 post-norm (GPT-1) */
  int32_t final_ln;    /* 1: apply ln_f before the head (pre-norm models); 0: none */
  int32_t gelu;        /* 0 tanh approximation, 1 exact erf form */
  int32_t dtype;       /* 0 fp32 SIMT parity mode, 1 bf16 tensor-core path (fp32 accumulation) */
  float ln_eps;        /* LayerNorm eps inside the square root, 1e-5 */
  int64_t max_tokens;  /* workspace bound: the largest B*T a forward call may use */
  int32_t untied_head; /* 0: the head is E itself (tied, "第 25 章" §25.4); 1: its own [V, C] matrix
                          (the MiniGPT page's nn.Linear(C, V) without bias) */
} gpt_config;

/* One block's parameters, all fp32, HOST memory, nn.Linear orientation. */
typedef struct gpt_layer_weights {
  const float* ln1_g;  const float* ln1_b;     /* [C], [C] */
  const float* attn_w; const float* attn_b;    /* c_attn  [3C, C], [3C] */
  const float* proj_w; const float* proj_b;    /* c_proj  [C, C],  [C]  */
  const float* ln2_g;  const float* ln2_b;     /* [C], [C] */
  const float* fc_w;   const float* fc_b;      /* c_fc    [ffn, C], [ffn] */
  const float* mp_w;   const float* mp_b;      /* mlp c_proj [C, ffn], [C] */
} gpt_layer_weights;

typedef struct gpt_weights {
  const float* wte;                  /* token table E [V, C]; also the head when tied */
  const float* wpe;                  /* position table P [ctx, C] */
  const gpt_layer_weights* layers;   /* L entries */
  const float* lnf_g;                /* [C]; may be NULL when final_ln == 0 */
  const float* lnf_b;
  const float* head;                 /* [V, C] head matrix when untied_head == 1, else ignored */
} gpt_weights;

typedef struct gpt_model gpt_model;

/*
 * Create a model on the current CUDA device.
 * cfg and weights are read during the call only: the library copies every
 * weight into library-owned device memory (bf16 for matrices and tables when
 * dtype == 1, fp32 otherwise; biases and LayerNorm parameters stay fp32), so
 * the caller may free its buffers on return. It also allocates the workspace
 * for cfg->max_tokens tokens and builds the TMA descriptors of the weights.
 * On success *out receives the handle; on failure *out is NULL and nothing leaks.
 * GPT_GB300_NO_PDL=1 in the environment (read once per process) launches the
 * kernels without Programmatic Dependent Launch overlap; the results are the
 * same bit for bit.
 */
int gpt_create(const gpt_config* cfg, const gpt_weights* weights, gpt_model** out);

/*
 * One forward pass and (if d_targets is non-NULL) the mean cross-entropy.
 *   d_ids      device int32 [B, T], row-major, values in [0, V)
 *   d_targets  device int32 [B, T] or NULL (then no loss is computed)
 *   d_loss     device fp32 scalar or NULL
 *   d_logits   device fp32 [B, T, V] or NULL; logits are written only when
 *              non-NULL (otherwise the head never writes them to memory)
 * Stream-ordered and asynchronous: host-checkable errors (pointers, shapes)
 * return immediately; device-found errors (token ids, targets, timeouts) are
 * recorded on the device and returned by the next gpt_status(). Calls on one
 * model share its workspace, so they must be ordered on one stream.
 * bf16 models capture the pass into a CUDA graph on the first call with a
 * given (pointers, B, T, armed probe) and replay it while those repeat
 * (GPT_GB300_NO_GRAPH=1 launches the kernels directly; same results).
 */
int gpt_forward(gpt_model* m, const int32_t* d_ids, const int32_t* d_targets, int32_t B,
                int32_t T, float* d_loss, float* d_logits, void* stream);

/*
 * The same forward pass from HOST buffers: copies h_ids/h_targets to the
 * device, runs gpt_forward, copies the loss (and logits if h_logits is
 * non-NULL) back, and synchronises the stream. Returns the device status too.
 * h_loss may be NULL only when h_targets is NULL.
 */
int gpt_forward_host(gpt_model* m, const int32_t* h_ids, const int32_t* h_targets, int32_t B,
                     int32_t T, float* h_loss, float* h_logits, void* stream);

/* Steps of the forward pass, for gpt_time_step(). */
enum {
  GPT_STEP_EMBED = 0,      /* embedding gather-add (+ first LayerNorm on pre-norm models) */
  GPT_STEP_C_ATTN = 1,     /* fused QKV projection of block `layer` */
  GPT_STEP_ATTN = 2,       /* causal attention of block `layer` */
  GPT_STEP_C_PROJ = 3,     /* attention output projection + residual */
  GPT_STEP_LN_MID = 4,     /* the LayerNorm between attention and MLP */
  GPT_STEP_C_FC = 5,       /* MLP up-projection + GELU */
  GPT_STEP_MLP_PROJ = 6,   /* MLP down-projection + residual */
  GPT_STEP_LN_OUT = 7,     /* the LayerNorm after the block (next ln_1, ln_f or post-norm ln_2) */
  GPT_STEP_HEAD = 8,       /* tied LM head (+ fused cross-entropy partials) */
  GPT_STEP_CE = 9,         /* cross-entropy combine */
  GPT_STEP_MEAN = 10,      /* mean of the per-position losses */
  /* steps of gpt_backward (its forward part uses the ids above) */
  GPT_STEP_B_DZ = 16,      /* cross-entropy gradient dz from the recomputed head logits */
  GPT_STEP_B_DH = 17,      /* dh = dz E */
  GPT_STEP_B_DE = 18,      /* the head's share of the table gradient, dz^T h */
  GPT_STEP_B_MP_W = 19,    /* block `layer`: weight gradient of the MLP down-projection */
  GPT_STEP_B_DG = 20,      /* dg = dx W_mp */
  GPT_STEP_B_FC_W = 21,    /* weight gradient of the MLP up-projection */
  GPT_STEP_B_DA2 = 22,     /* du W_fc */
  GPT_STEP_B_PROJ_W = 23,  /* weight gradient of the attention output projection */
  GPT_STEP_B_DY = 24,      /* dy = ds1 W_proj */
  GPT_STEP_B_ATTN = 25,    /* causal attention derivative (two kernels) */
  GPT_STEP_B_ATTN_W = 26,  /* weight gradient of the QKV projection */
  GPT_STEP_B_DA1 = 27      /* dqkv W_attn */
};

/*
 * Arm a timing probe for the NEXT gpt_forward (or gpt_backward) on this model: ev_start
 * (cudaEvent_t) is recorded on the forward's stream just before the kernel of
 * `step` (in block `layer`; ignored for steps outside the blocks) and ev_stop
 * just after it. The probe disarms after that forward. Pass ev_start == NULL
 * to disarm. On the graph-replayed bf16 forward the two records are nodes of
 * the graph; a later call with the same (step, layer) points them at its own
 * events when the driver accepts those events for that (events from
 * cudaEventCreate do; PyTorch's are refused), else it captures the pass again
 * (correct, but slower by the capture). A failed record returns GPT_ECUDA.
 */
int gpt_time_step(gpt_model* m, int step, int layer, void* ev_start, void* ev_stop);

/* Number of kernels the last gpt_forward call launched (0 before the first). */
int gpt_last_launch_count(const gpt_model* m);

/* Number of launches the probe armed for the last gpt_forward bracketed: 1, or
 * 0 when that step did not run (the loss steps of a forward without targets, a
 * block index past the last block). */
int gpt_last_probe_hits(const gpt_model* m);

/*
 * Failure-detection check of the bounded device waits (the pages have no
 * counterpart: it tests the library's own error path). Arms the next bf16
 * gpt_forward on m, which then runs with direct launches (no graph): in the
 * long-K projections whose tiles are split between two CTAs (stream-K), each
 * CTA that finishes a split tile waits on a partial-tile flag that nothing sets,
 * for at most limit_cycles SM clock cycles (about limit_cycles / 2e9 seconds)
 * instead of about 2 s. Every such wait expires: the kernel records a device
 * error, raises its CTA's abort flag, drains its own copies and MMAs, frees its
 * tensor memory and returns. The loss of that call is unspecified; the next
 * gpt_status() returns GPT_EDEVICE and clears the flags the aborted launches
 * left set, after which the handle computes correct results again. A forward
 * with no split tiles is unaffected. The first call allocates a small flag
 * buffer. GPT_ECONFIG for fp32 models, GPT_EINVAL for limit_cycles < 1.
 */
int gpt_debug_expire_waits(gpt_model* m, int64_t limit_cycles);

/*
 * Incremental decoding with a key/value cache ("预训练一个 Mini GPT", the
 * sections on the KV cache and on prefill and decode: the keys and values of
 * every processed token are kept, so a new token costs one projection of its
 * own row per layer plus attention over the cached rows). bf16 models only
 * (GPT_ECONFIG otherwise).
 *
 * gpt_kv_reserve: allocate (or grow) the model-owned cache for up to
 * max_batch sequences of ctx tokens: L x max_batch x ctx x 2C bf16
 * (604 MB for GPT-2 small at 16 sequences). Synchronous; GPT_ENOMEM on failure.
 * Growing the cache discards the rows it held.
 */
int gpt_kv_reserve(gpt_model* m, int32_t max_batch);

/*
 * Prefill: the forward pass over prompts d_ids [B, T] (device int32, all of
 * length T) that also stores every token's key and value in the cache (rows
 * 0..T-1 of sequences 0..B-1), and writes the logits of each sequence's last
 * token to d_logits [B, V] (device fp32; NULL: not computed). Requires
 * B <= the reserved batch (GPT_EINVAL), T <= ctx (GPT_ESEQ), B*T <= max_tokens.
 * Stream-ordered and asynchronous like gpt_forward.
 */
int gpt_prefill(gpt_model* m, const int32_t* d_ids, int32_t B, int32_t T, float* d_logits, void* stream);

/*
 * One decode step: token d_ids[b] (device int32 [B]) is appended to sequence
 * b at position pos (its key and value go to cache row pos; rows 0..pos-1
 * must hold that sequence's earlier tokens, from gpt_prefill and earlier
 * steps), and d_logits [B, V] (device fp32) receives the next-token logits,
 * equal to row pos of a full forward over the sequence. Requires
 * 0 <= pos < ctx (GPT_ESEQ) and B <= the reserved batch (GPT_EINVAL).
 * Stream-ordered and asynchronous; bad ids are reported by gpt_status().
 * The step's kernels are captured into a CUDA graph on the first call for a
 * given (B, d_logits) and replayed afterwards (the ids and the position are
 * read from model memory); GPT_GB300_NO_GRAPH=1 launches them directly.
 */
int gpt_decode_step(gpt_model* m, const int32_t* d_ids, int32_t B, int32_t pos, float* d_logits, void* stream);

/*
 * Next-token draw for each row of d_logits [B, V] (device fp32, row stride V)
 * ("预训练一个 Mini GPT" 第7步 text generation; "02 GPT 架构" 8.1-8.3):
 * temperature <= 0 is greedy (the most probable token, the lowest index among
 * equal maxima); otherwise probabilities softmax(logits / temperature), then
 * top_k (> 0 and < V: keep the k most probable), then top_p (in (0, 1): keep
 * the smallest leading set, by probability then index, whose mass reaches
 * top_p of the kept mass), renormalise, and take the first index (in index
 * order) whose cumulative probability exceeds d_uniform[b] (device fp32 [B],
 * values in [0, 1), drawn by the caller). Writes d_ids [B] (device int32).
 * Requires 1 <= V <= 55296 (the row's probabilities are held on chip).
 * Stream-ordered and asynchronous; model-independent.
 */
int gpt_sample(const float* d_logits, int32_t B, int32_t V, float temperature, int32_t top_k, float top_p,
               const float* d_uniform, int32_t* d_ids, void* stream);

/*
 * Back-propagation of the mean next-token cross-entropy ("预训练一个 Mini GPT",
 * 训练循环: forward, loss, then the gradient of every parameter), bf16 models
 * only (GPT_ECONFIG otherwise). Runs the forward pass and loss (d_loss, device
 * fp32, nullable) on ids and targets (device int32 [B, T]), then writes the
 * gradient of that loss with respect to every parameter into model-owned fp32
 * buffers, overwriting the previous call's. The tied token table's gradient
 * is the sum of its embedding and head shares ("第 25 章 从小 GPT 到 GPT-2"
 * §25.4). T <= ctx (GPT_ESEQ), B*T <= max_tokens (GPT_EINVAL). The first call allocates the workspace synchronously:
 * every block's activations at max_tokens, the gradients, transposed weights
 * and the head's dz (about 11 GB for GPT-2 small at 16384 tokens; GPT_ENOMEM
 * on failure); later
 * calls are stream-ordered. Token and target errors are reported by
 * gpt_status, as for gpt_forward.
 */
int gpt_backward(gpt_model* m, const int32_t* d_ids, const int32_t* d_targets, int32_t B, int32_t T,
                 float* d_loss, void* stream);

/* Parameters, for gpt_grad (the per-block ones take a layer index). */
enum {
  GPT_P_WTE = 0, GPT_P_WPE = 1, GPT_P_LNF_G = 2, GPT_P_LNF_B = 3,
  GPT_P_LN1_G = 4, GPT_P_LN1_B = 5, GPT_P_ATTN_W = 6, GPT_P_ATTN_B = 7,
  GPT_P_PROJ_W = 8, GPT_P_PROJ_B = 9, GPT_P_LN2_G = 10, GPT_P_LN2_B = 11,
  GPT_P_FC_W = 12, GPT_P_FC_B = 13, GPT_P_MP_W = 14, GPT_P_MP_B = 15,
  GPT_P_HEAD = 16                    /* the untied head's matrix (GPT_EINVAL on tied models) */
};

/*
 * The device pointer (fp32, model-owned, laid out as the weight: [out, in]
 * for the matrices) and element count of one parameter's gradient from the
 * last gpt_backward. GPT_EINVAL before the first gpt_backward or for an
 * unknown parameter or layer. Models without a final LayerNorm report zeros
 * for GPT_P_LNF_G / GPT_P_LNF_B.
 */
int gpt_grad(const gpt_model* m, int param, int layer, float** d_grad, int64_t* numel);

/* Copies that gradient into caller device memory d_dst (numel fp32 values), stream-ordered. */
int gpt_grad_copy(const gpt_model* m, int param, int layer, float* d_dst, void* stream);

/*
 * One AdamW step on every parameter from the last gpt_backward's gradients
 * ("Day 16 从零组装 MiniGPT": loss, backward, AdamW, parameters change;
 * "预训练一个 Mini GPT" 训练循环): p -= lr wd p (weight matrices and the two
 * tables only), m = b1 m + (1 - b1) g, v = b2 v + (1 - b2) g^2,
 * p -= lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps), t counting calls
 * from 1. The model keeps fp32 master weights and both moments (allocated
 * synchronously by the first call, 3 x 4 bytes per parameter; GPT_ENOMEM on
 * failure) and writes the updated values into its own weights (bf16 matrices
 * rounded to nearest). GPT_EINVAL before the first gpt_backward or for betas
 * outside [0, 1) or eps <= 0. Stream-ordered.
 */
int gpt_adamw_step(gpt_model* m, float lr, float beta1, float beta2, float eps, float weight_decay, void* stream);

/* Copies one parameter's fp32 master weight (after a gpt_adamw_step) into d_dst. GPT_EINVAL before. */
int gpt_master_copy(const gpt_model* m, int param, int layer, float* d_dst, void* stream);

/* Synchronise the stream, read and clear the model's device error word. */
int gpt_status(gpt_model* m, void* stream);

/* Free everything the model owns. Safe on NULL. */
void gpt_destroy(gpt_model* m);

/* Static description of a status code. */
const char* gpt_strerror(int code);

/* Text of the last failing CUDA call made by this thread inside the library
 * (empty if none); valid until the thread's next library call. */
const char* gpt_last_error_detail(void);

/* Unique parameter count of cfg with the tied head ("第 25 章" §25.4). */
int64_t gpt_param_count(const gpt_config* cfg);

#ifdef __cplusplus
}
#endif

#endif /* GPT_GB300_H */
