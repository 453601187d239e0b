/*
 * gpt2fwd.h -- C ABI of the GPT-2 forward-pass library for one NVIDIA GB300
 * (sm_103a).  Library file: libgpt2fwd.so.
 *
 * Sources of the operations (web pages the method is taken from):
 *   [ECE408]  "ECE408 Final Project - GPT-2", Milestone 1 README: section
 *             "Milestone Requirements" (host functions `xxxx_forward()` only
 *             launch kernels; the caller allocates and copies memory; their
 *             signatures are fixed, the kernels are free) and the grade table
 *             of "Code Submission and Grading" (the forward-pass kernels:
 *             Attention including Softmax, Encoder, LayerNorm, MatMul,
 *             Residual, GELU).
 *   [llm.c]   "State of the Union [April 22, 2024]" (llm.c discussion #224):
 *             the per-kernel table naming the forward kernels
 *             (encoder_forward, layernorm_forward, the attention softmax,
 *             gelu_forward, residual_forward, the classifier) and the GEMMs.
 *   [NTU]     NTU optdl2025 project list: "Understanding and Improving GPT-2
 *             Implementations in NanoGPT" (fused QKV projection, heads split
 *             as column blocks, KV caching for autoregressive prediction) and
 *             "Understand FlashAttention (I)" (Algorithms 0 and 1: exact
 *             attention with a tiled online softmax).
 *
 * Conventions shared by every call:
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     the argument says "host".  No call allocates, frees or copies memory
 *     between host and device.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work on it and return without synchronising.
 *   - Floating-point tensors are IEEE fp32, row-major, unless a precision
 *     mode below says otherwise for an internal buffer.
 *   - Return value: GPT2_OK (0) or a negative GPT2_ERR_* code.  Arguments are
 *     checked on the host before anything is enqueued; on error nothing is
 *     enqueued.  Faults found on the device (a token id outside [0, V), a
 *     pipeline wait that gave up) never trap: they set a device error word
 *     read by gpt2_get_error().
 *   - Pointers must be 16-byte aligned (128-bit vector accesses).
 */
#ifndef GPT2FWD_H
#define GPT2FWD_H

#include <stddef.h>

#if defined(__GNUC__)
#define GPT2_API __attribute__((visibility("default")))
#else
#define GPT2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Model hyper-parameters (GPT-2 names maxT, V, Vp, L, NH, C). */
typedef struct {
  int max_seq_len;       /* maxT: longest sequence, size of the position table */
  int vocab_size;        /* V: number of real tokens */
  int padded_vocab_size; /* Vp >= V: rows of the token embedding and logits columns */
  int num_layers;        /* L */
  int num_heads;         /* NH; head size hs = C / NH */
  int channels;          /* C */
} GPT2Config;

/* Operand precision of the matrix products (GEMMs and attention).
 *   GPT2_FP32: fp32 CUDA-core arithmetic throughout (reference-grade mode).
 *   GPT2_TF32: tensor cores (tcgen05 kind::tf32) on fp32 operands; the
 *              attention runs the bf16 tensor-core kernel.
 *   GPT2_BF16: tensor cores (tcgen05 kind::f16) on bf16 operands.
 *   GPT2_FP16: tensor cores (tcgen05 kind::f16) on fp16 operands: the same
 *              rate as bf16 with 8x finer rounding (11 significant bits
 *              against 8) and a range of +-65504, ample for GPT-2's
 *              normalised activations and 0.02-scale weights.
 * In the 16-bit modes the operand buffers internal to gpt2_forward (and
 * the KV cache) hold the 16-bit type, since the tensor cores would round
 * them to it anyway, and so do the attention and MLP projections' outputs
 * before the residual add (performed in the LayerNorm that follows); the
 * residual stream, logits and probabilities stay fp32.  Accumulation is
 * fp32 in every mode. */
typedef enum { GPT2_FP32 = 0, GPT2_TF32 = 1, GPT2_BF16 = 2, GPT2_FP16 = 3 } GPT2Precision;

/* Element type of a probabilities output (softmax_forward_ex,
 * gpt2_forward_ex, gpt2_forward_profile) [llm.c "State of the Union": the
 * classifier row of its kernel table, and its case for fp16/bf16 storage].
 * GPT2_PROBS_F32 is the default of softmax_forward and gpt2_forward; the
 * 16-bit types hold each fp32 probability rounded to nearest once (so they
 * equal the fp32 output rounded) and halve the bytes of the largest write of
 * the forward pass. */
typedef enum { GPT2_PROBS_F32 = 0, GPT2_PROBS_F16 = 1, GPT2_PROBS_BF16 = 2 } GPT2ProbsType;

enum {
  GPT2_OK = 0,
  GPT2_ERR_ARG = -1,       /* null pointer or nonsensical argument */
  GPT2_ERR_SHAPE = -2,     /* T > maxT, C % NH, pos >= maxT, unsupported shape */
  GPT2_ERR_ALIGN = -3,     /* pointer not 16-byte aligned */
  GPT2_ERR_WORKSPACE = -4, /* workspace or buffer too small */
  GPT2_ERR_CUDA = -5,      /* a CUDA runtime call or launch failed */
  GPT2_ERR_DEVICE = -6,    /* device-detected fault (see gpt2_get_error) */
  GPT2_ERR_UNSUPPORTED = -7
};

/* Device error word bits returned by gpt2_get_error (as -GPT2_ERR_DEVICE
 * combined into a positive bit set, see below). */
#define GPT2_DEVERR_TOKEN_BIT 1    /* token id outside [0, V); the read was clamped */
#define GPT2_DEVERR_TIMEOUT_BIT 2  /* a pipeline wait gave up after ~1 s */
#define GPT2_DEVERR_POSITION_BIT 4 /* a decode position outside [0, maxT) or past its sequence's blocks */
#define GPT2_DEVERR_BLOCK_BIT 8    /* a block-table entry outside [0, num_blocks); read as block 0 */

/* ----------------------------------------------------------- single steps */

/* Encoder [ECE408 grade table "Encoder"; llm.c table encoder_forward]:
 *   out[b,t,c] = wte[tok[b,t], c] + wpe[t, c]
 * out [B,T,C] fp32, tok [B,T] int32, wte [V',C] (any V' >= V rows), wpe
 * [>=T, C].  A token outside [0, V) is clamped to 0 for the read and flags
 * GPT2_DEVERR_TOKEN_BIT.  Requires C % 4 == 0. */
GPT2_API int encoder_forward(float* out, const int* tok, const float* wte, const float* wpe, int B, int T, int C, int V,
                    void* stream);

/* LayerNorm [ECE408 "LayerNorm"; llm.c layernorm_forward]: per row of C
 *   mean = sum x / C, var = sum (x - mean)^2 / C, rstd = 1/sqrt(var + 1e-5),
 *   out = (x - mean) * rstd * w + b.
 * out, inp [N,C]; w, b [C]; mean and rstd [N] are written when non-null.
 * Requires C % 4 == 0.  out may alias inp. */
GPT2_API int layernorm_forward(float* out, float* mean, float* rstd, const float* inp, const float* w, const float* b, int N,
                      int C, void* stream);

/* Scratch bytes matmul_forward needs for this shape and precision (0 for
 * GPT2_FP32 and GPT2_TF32; the 16-bit copies of inp and W for GPT2_BF16 and
 * GPT2_FP16). */
GPT2_API size_t matmul_workspace_size(int N, int C, int OC, int precision);

/* MatMul with bias [ECE408 "MatMul"; llm.c GEMMs]:
 *   out[n, o] = sum_k inp[n, k] * W[o, k] + bias[o]     (bias may be NULL)
 * out [N,OC], inp [N,C], W [OC,C] (PyTorch Linear layout), bias [OC].
 * Tensor-core modes need C % 8 == 0 and OC % 4 == 0.  `workspace` of
 * matmul_workspace_size() bytes is caller-owned scratch (may be NULL when
 * that size is 0).  out must not alias inp or W.  In the tensor-core modes
 * N <= 64 rows (a decode step's shape) run on a kernel that splits C over
 * the CTAs of a cluster and adds the parts in a fixed order: repeated calls
 * give identical results, which may differ in the last bits from the same
 * rows computed inside a larger N. */
GPT2_API int matmul_forward(float* out, const float* inp, const float* W, const float* bias, int N, int C, int OC,
                   int precision, void* workspace, size_t ws_bytes, void* stream);

/* matmul_forward without a caller workspace, for callers that cannot
 * allocate device memory (code that must not call cudaMalloc because it can
 * synchronise the device, or a plugin inside a program that owns every
 * device allocation and offers it no workspace).  The pages have no
 * counterpart of this call; it exists for such callers only.
 * Arguments, layouts and results are those of matmul_forward.  The 16-bit
 * copies that the GPT2_BF16 and GPT2_FP16 modes need live in a fixed 16 MiB
 * device array inside the library (every GPU that loads the library holds
 * it until the process exits): shapes with matmul_workspace_size(N, C, OC,
 * precision) > 16 MiB are rejected with GPT2_ERR_WORKSPACE.  GPT2_FP32 and
 * GPT2_TF32 need no scratch.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All
 * calls share the one array and each overwrites it before reading it, so
 * calls whose work overlaps on the GPU (on different streams, or different
 * host threads without ordering) race and give wrong results: order them on
 * one stream.  Allocates nothing: no cudaMalloc, cudaFree or allocating
 * library routine is called. */
GPT2_API int matmul_forward_noalloc(float* out, const float* inp, const float* W, const float* bias, int N, int C,
                                   int OC, int precision, void* stream);

/* Scratch bytes attention_forward needs (the 16-bit copy of qkv in the
 * tensor-core modes, 0 in GPT2_FP32). */
GPT2_API size_t attention_workspace_size(int B, int T, int C, int precision);

/* Causal multi-head attention including its softmax [ECE408 "Attention
 * (including Softmax)"; NTU NanoGPT head splitting; FlashAttention
 * Algorithm 0 defines the result, Algorithm 1's online softmax computes it]:
 *   q, k, v = columns [0,C), [C,2C), [2C,3C) of qkv; head h owns columns
 *   [h*hs, (h+1)*hs) of each; S = q k^T / sqrt(hs) with keys j <= t only;
 *   out[b,t, h*hs:(h+1)*hs] = softmax_j(S[t, :]) v.
 * out [B,T,C], qkv [B,T,3C].  Requires hs in {16, 32, 64}.  GPT2_FP32
 * runs fp32 CUDA-core arithmetic; the tensor-core modes round Q, K, V and
 * the probabilities to the 16-bit type (bf16 for GPT2_TF32 and GPT2_BF16,
 * fp16 for GPT2_FP16) of a copy of qkv made in `workspace`, and accumulate
 * in fp32. */
GPT2_API int attention_forward(float* out, const float* qkv, int B, int T, int C, int NH, int precision, void* workspace,
                      size_t ws_bytes, void* stream);

/* Scratch bytes attention_backward needs at this precision; 0 for a
 * precision or head size it does not support.  GPT2_FP32: two [B][NH][T]
 * fp32 arrays (the forward's per-row softmax statistic and rowsum(dout *
 * out)).  GPT2_TF32 / GPT2_BF16 (head size 64): bf16 copies of qkv and dout,
 * a bf16 [B,T,C] scratch output and two [B][NH][Tp] fp32 arrays (Tp = T
 * rounded up to 128). */
GPT2_API size_t attention_backward_workspace_size(int B, int T, int C, int NH, int precision);

/* The backward pass of causal multi-head attention ["Understand
 * FlashAttention (II)": the backward algorithms of Algorithms 0 and 1; the
 * llm.c table's attention backward kernels]:
 *   with S = q k^T / sqrt(hs) (causal), P = softmax_rows(S), out = P v and
 *   dout = dL/dout:  dv = P^T dout,  dP = dout v^T,
 *   dS = P (dP - rowsum(dout * out)),  dq = dS k / sqrt(hs),
 *   dk = dS^T q / sqrt(hs),
 * per (sequence, head), written into dqkv [B,T,3C] in the column blocks of
 * q, k and v (every element written).  qkv [B,T,3C] and out [B,T,C] are
 * the forward's input and output, dout [B,T,C].  P is recomputed tile by
 * tile from a per-row statistic, never stored; the results do not depend
 * on timing.
 *   GPT2_FP32: fp32 CUDA-core arithmetic, hs in {16, 32, 64}; the statistic
 *     is recomputed from qkv.
 *   GPT2_TF32, GPT2_BF16: tcgen05 tensor cores, hs = 64: q, k, v, dout, P
 *     and dS rounded to bf16, fp32 accumulation; the statistic comes from a
 *     run of the tensor-core forward (its output discarded), rowsum(dout *
 *     out) from the given fp32 out.
 *   GPT2_FP16 (and another hs in a 16-bit mode): GPT2_ERR_UNSUPPORTED.
 * Workspace of attention_backward_workspace_size bytes, 16-byte aligned. */
GPT2_API int attention_backward(float* dqkv, const float* dout, const float* qkv, const float* out, int B, int T,
                                int C, int NH, int precision, void* workspace, size_t ws_bytes, void* stream);

/* tanh-GELU [ECE408 "GELU"; llm.c gelu_forward]:
 *   out = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), n elements. */
GPT2_API int gelu_forward(float* out, const float* inp, int n, void* stream);

/* Residual [ECE408 "Residual"; llm.c residual_forward]: out = a + b, n
 * elements; out may alias a or b. */
GPT2_API int residual_forward(float* out, const float* a, const float* b, int n, void* stream);

/* Softmax over the vocabulary [llm.c classifier; the final logits softmax]:
 *   probs[n, v] = exp(l[n,v] - max_u l[n,u]) / sum_{u<V} exp(l[n,u] - max)
 * for v < V, and probs[n, v] = 0 for V <= v < Vp.  logits, probs [N,Vp];
 * requires Vp % 4 == 0.  probs must not alias logits. */
GPT2_API int softmax_forward(float* probs, const float* logits, int N, int V, int Vp, void* stream);

/* softmax_forward with the probabilities stored as probs_type (a
 * GPT2ProbsType): probs [N,Vp] of that type, 16-byte aligned; a
 * probs_type outside GPT2ProbsType is GPT2_ERR_ARG. */
GPT2_API int softmax_forward_ex(void* probs, int probs_type, const float* logits, int N, int V, int Vp,
                                void* stream);

/* Greedy next token: next[b] = the smallest v < V with the largest
 * logits[b, v].  next [B] int32, logits [B,Vp]. */
GPT2_API int gpt2_argmax(int* next, const float* logits, int B, int V, int Vp, void* stream);

/* ------------------------------------------------------ the forward pass */

/* Number of fp32 values in the flat parameter buffer.  Tensor order, each
 * row-major: wte[Vp,C] wpe[maxT,C] ln1w[L,C] ln1b[L,C] qkvw[L,3C,C]
 * qkvb[L,3C] attprojw[L,C,C] attprojb[L,C] ln2w[L,C] ln2b[L,C] fcw[L,4C,C]
 * fcb[L,4C] fcprojw[L,C,4C] fcprojb[L,C] lnfw[C] lnfb[C]. */
GPT2_API size_t gpt2_num_parameters(const GPT2Config* cfg);

/* Bytes of the packed weight buffer for a precision: 16-bit copies of the
 * matrices (wte, qkvw, attprojw, fcw, fcprojw) for GPT2_BF16 and
 * GPT2_FP16, 0 otherwise. */
GPT2_API size_t gpt2_packed_weights_size(const GPT2Config* cfg, int precision);

/* Fills `packed` (caller-owned, gpt2_packed_weights_size bytes) from the
 * fp32 parameters.  Run once per set of weights; gpt2_forward and
 * gpt2_decode_step read it in the 16-bit modes. */
GPT2_API int gpt2_prepare_weights(const GPT2Config* cfg, const float* params, void* packed, size_t bytes, int precision,
                         void* stream);

/* Scratch bytes gpt2_forward / gpt2_decode_step need for B sequences of T
 * tokens (use T = 1 for decode). */
GPT2_API size_t gpt2_workspace_size(const GPT2Config* cfg, int B, int T, int precision);

/* Bytes of a KV cache for B sequences: layout [L][2][B][NH][maxT][hs]
 * (keys then values per layer), fp32 in GPT2_FP32 / GPT2_TF32, the 16-bit
 * type in GPT2_BF16 / GPT2_FP16. */
GPT2_API size_t gpt2_kvcache_size(const GPT2Config* cfg, int B, int precision);

/* The GPT-2 forward pass (pre-LayerNorm blocks) over B sequences of T
 * tokens [ECE408 Introduction: the forward pass; llm.c: encoder, forward
 * blocks, classifier]:
 *   x = encoder(tok); for each layer l:
 *     x += attproj(attention(qkv(LN1(x))));  x += fcproj(GELU(fc(LN2(x))))
 *   logits = LN_f(x) wte^T (tied, no bias; all Vp columns);
 *   probs  = softmax over the first V columns (when probs != NULL).
 * params: flat fp32 buffer (gpt2_num_parameters values, never written);
 * packed: output of gpt2_prepare_weights (required in the 16-bit modes,
 * else ignored); tok [B,T] int32; logits [B,T,Vp]; probs [B,T,Vp] or NULL;
 * kvcache: NULL, or a cache of gpt2_kvcache_size(cfg, B, precision) bytes
 * whose positions [0, T) are written (the prefill of decoding);
 * workspace of gpt2_workspace_size(cfg, B, T, precision) bytes.
 * Requires 1 <= T <= maxT and C % NH == 0.  In the 16-bit modes the pass's
 * kernels are programmatic dependent launches: each may begin its set-up
 * while the kernel ahead of it on the stream runs and waits for that kernel
 * before touching what it writes, so stream order holds for the caller's
 * own work before and after the call. */
GPT2_API int gpt2_forward(const GPT2Config* cfg, const float* params, const void* packed, const int* tok, int B, int T,
                 float* logits, float* probs, void* kvcache, void* workspace, size_t ws_bytes, int precision,
                 void* stream);

/* gpt2_forward with the probabilities stored as probs_type (a
 * GPT2ProbsType): probs [B,T,Vp] of that type (16-byte aligned) or NULL;
 * the logits stay fp32.  A probs_type outside GPT2ProbsType is
 * GPT2_ERR_ARG.  Other arguments and behaviour as gpt2_forward. */
GPT2_API int gpt2_forward_ex(const GPT2Config* cfg, const float* params, const void* packed, const int* tok, int B,
                             int T, float* logits, void* probs, int probs_type, void* kvcache, void* workspace,
                             size_t ws_bytes, int precision, void* stream);

/* One KV-cached decode step [NTU "KV Caching"]: each of the B sequences has
 * `pos` tokens in kvcache (positions [0, pos)) and gets one new token
 * tok[b] at position pos.  Writes this position's keys and values into the
 * cache and computes logits [B,Vp] (and probs [B,Vp] when non-null) exactly
 * as row `pos` of gpt2_forward over the whole sequence would.  Requires
 * 0 <= pos < maxT; workspace of gpt2_workspace_size(cfg, B, 1, precision).
 * The new keys and values are appended by the attention kernel.  In the
 * 16-bit modes the step's kernels are programmatic dependent launches: each
 * may begin (set up, request weights) while the kernel ahead of it on the
 * stream runs, and waits for it before touching what it writes, so stream
 * order holds for the caller's own work before and after the call. */
GPT2_API int gpt2_decode_step(const GPT2Config* cfg, const float* params, const void* packed, void* kvcache, const int* tok,
                     int B, int pos, float* logits, float* probs, void* workspace, size_t ws_bytes, int precision,
                     void* stream);

/* ------------------------------------------------------- training step */

/* Workspace bytes of gpt2_forward_backward for B sequences of T tokens
 * (every layer's fp32 activations and the backward's scratch); 0 unless
 * precision is GPT2_FP32 or GPT2_TF32. */
GPT2_API size_t gpt2_train_workspace_size(const GPT2Config* cfg, int B, int T, int precision);

/* The loss and gradient of one training step [llm.c "State of the Union":
 * a GPT-2 training step is the forward blocks, the classifier (softmax with
 * cross-entropy), the backward blocks and the optimizer; its per-kernel
 * table names the backward kernels built here: matmul backward with its
 * bias, layernorm backward, gelu backward, attention backward, encoder
 * backward]:
 *   loss = mean over the B*T positions of -log softmax(logits)[target],
 *          the softmax over the first V columns (loss: DEVICE, one float);
 *   grads = dloss/dparams, in the layout of the flat parameter buffer
 *          (gpt2_num_parameters floats, DEVICE, every element written).
 * params as gpt2_forward's (fp32, never written); tok, targets [B,T] int32
 * (DEVICE).  Activations and gradients are fp32; the matmuls (and their
 * backward products) run on fp32 CUDA cores in GPT2_FP32 and on tcgen05
 * tensor cores with tf32 operands in GPT2_TF32 (then B*T % 4 == 0); the
 * attention's forward runs in fp32 on CUDA cores in GPT2_FP32 and on the
 * bf16 tensor-core kernel in GPT2_TF32 (as gpt2_forward's tf32 mode), its
 * backward in fp32 on CUDA cores in both.
 * Other precisions return GPT2_ERR_UNSUPPORTED.  The token-embedding
 * gradient sums repeated tokens with atomics: its last bits can vary from
 * run to run; every other element is deterministic.  A target outside
 * [0, V) sets GPT2_DEVERR_TOKEN_BIT. */
GPT2_API int gpt2_forward_backward(const GPT2Config* cfg, const float* params, float* grads, const int* tok,
                                   const int* targets, int B, int T, float* loss, void* workspace, size_t ws_bytes,
                                   int precision, void* stream);

/* One AdamW step over n fp32 values [llm.c "State of the Union": the
 * optimizer of the training step; the update is AdamW's, decoupled weight
 * decay (Loshchilov and Hutter), the same decay for every parameter]:
 *   m = beta1 m + (1 - beta1) g,  v = beta2 v + (1 - beta2) g^2,
 *   params -= lr (m / (1 - beta1^t) / (sqrt(v / (1 - beta2^t)) + eps)
 *                 + weight_decay params),
 * t >= 1 the step number; m and v (DEVICE, n floats each, zero before the
 * first step) are updated in place. */
GPT2_API int gpt2_adamw(float* params, const float* grads, float* m, float* v, size_t n, float lr, float beta1,
                        float beta2, float eps, float weight_decay, int t, void* stream);

/* --------------------------------------------------- paged KV cache */

/* A paged KV cache [NTU "KV Caching": the keys and values of earlier
 * positions are kept and reused, not recomputed].  Instead of one dense
 * [maxT] slab per sequence, positions live in fixed-size blocks of a shared
 * pool, found through a per-sequence block table, so that sequences of
 * different lengths share one allocation and a sequence holds only the
 * blocks it uses.
 *   pool:        DEVICE, gpt2_paged_kvcache_size(cfg, num_blocks,
 *                block_size, precision) bytes, 16-byte aligned; layout
 *                [L][2][num_blocks][NH][block_size][hs] (per layer the key
 *                blocks, then the value blocks), element type as the dense
 *                cache's (fp32, or the 16-bit type in GPT2_BF16/GPT2_FP16);
 *   block_table: DEVICE int32 [B][max_blocks_per_seq]: position p of
 *                sequence b is in block block_table[b][p / block_size],
 *                slot p % block_size.  Entries a call never reaches may hold
 *                anything; an entry it reaches outside [0, num_blocks) sets
 *                GPT2_DEVERR_BLOCK_BIT (block 0 is used instead).
 *   block_size:  positions per block, a power of two;
 *   max_blocks_per_seq: row length of block_table, 1 .. 1024.
 * A sequence can hold min(maxT, max_blocks_per_seq * block_size)
 * positions.  The library never writes block_table; the caller owns the
 * pool, the table and the assignment of blocks to sequences. */
typedef struct {
  void* pool;
  const int* block_table;
  int num_blocks;
  int block_size;
  int max_blocks_per_seq;
} GPT2PagedKVCache;

/* Bytes of a paged pool of num_blocks blocks (0 for invalid arguments). */
GPT2_API size_t gpt2_paged_kvcache_size(const GPT2Config* cfg, int num_blocks, int block_size, int precision);

/* gpt2_forward that writes the keys and values of positions [0, T) of each
 * sequence into the paged cache `kv` (the prefill of paged decoding); the
 * outputs are gpt2_forward's.  Prompts of different lengths can share one
 * call padded to T: each sequence's later decode steps start at its own
 * length and overwrite the padded positions.  Requires T <= the capacity
 * of a sequence.  Other arguments as gpt2_forward. */
GPT2_API int gpt2_prefill_paged(const GPT2Config* cfg, const float* params, const void* packed, const int* tok, int B,
                                int T, float* logits, float* probs, const GPT2PagedKVCache* kv, void* workspace,
                                size_t ws_bytes, int precision, void* stream);

/* One KV-cached decode step over a paged cache [NTU "KV Caching"], each
 * sequence at its own position: sequence b has pos[b] positions cached and
 * gets token tok[b] at position pos[b] (pos: DEVICE int32 [B]).  Writes
 * that position's keys and values through the block table and computes
 * logits [B,Vp] (probs [B,Vp] when non-null) exactly as row pos[b] of
 * gpt2_forward over that sequence would.  A pos[b] outside [0, capacity)
 * sets GPT2_DEVERR_POSITION_BIT and leaves the cache unwritten (that row's
 * results are not meaningful).  Workspace: gpt2_workspace_size(cfg, B, 1,
 * precision).  Launch behaviour as gpt2_decode_step. */
GPT2_API int gpt2_decode_step_paged(const GPT2Config* cfg, const float* params, const void* packed,
                                    const GPT2PagedKVCache* kv, const int* tok, const int* pos, int B, float* logits,
                                    float* probs, void* workspace, size_t ws_bytes, int precision, void* stream);

/* ------------------------------------------------------------ diagnostics */

/* Stages of the forward pass, for gpt2_forward_profile. */
enum {
  GPT2_STAGE_ENCODER = 0,
  GPT2_STAGE_LN1 = 1,       /* all L layers summed, likewise below; in the
                               16-bit modes LN1 of layers 1.. and LN2 and
                               LN_f also add the preceding projection's
                               output into the residual stream */
  GPT2_STAGE_QKV = 2,       /* QKV GEMM (+ cache store when a prefill fills a cache) */
  GPT2_STAGE_ATTENTION = 3,
  GPT2_STAGE_ATTPROJ = 4,   /* attention projection GEMM (+ residual in the fp32 and tf32 modes) */
  GPT2_STAGE_LN2 = 5,
  GPT2_STAGE_FC = 6,        /* MLP up-projection GEMM + GELU */
  GPT2_STAGE_FCPROJ = 7,    /* MLP down-projection GEMM (+ residual in the fp32 and tf32 modes) */
  GPT2_STAGE_LNF = 8,
  GPT2_STAGE_LMHEAD = 9,
  GPT2_STAGE_SOFTMAX = 10,
  GPT2_NUM_STAGES = 11
};

/* gpt2_forward_ex (without a KV cache) with a CUDA event recorded on
 * `stream` after every stage; waits for the pass to finish and ADDS each
 * stage's milliseconds into stage_ms (HOST array of n_stages floats, indexed
 * by GPT2_STAGE_*).  probs of probs_type (a GPT2ProbsType) or NULL.  For
 * measurement only: the events serialise nothing but the call synchronises
 * the stream. */
GPT2_API int gpt2_forward_profile(const GPT2Config* cfg, const float* params, const void* packed, const int* tok,
                                  int B, int T, float* logits, void* probs, int probs_type, void* workspace,
                                  size_t ws_bytes, int precision, void* stream, float* stage_ms, int n_stages);

/* Synchronises `stream`, returns the device error word (a set of
 * GPT2_DEVERR_*_BIT bits, 0 when clean) and clears it; a negative
 * GPT2_ERR_CUDA if the synchronisation itself failed. */
GPT2_API int gpt2_get_error(void* stream);

/* Static text for a GPT2_ERR_* code. */
GPT2_API const char* gpt2_strerror(int code);

/* Text of the last CUDA error seen by the library on this host thread. */
GPT2_API const char* gpt2_last_cuda_error(void);

/* Runs the kernels' bounded-wait path once, on purpose, so that it can be
 * tested: one CTA waits on an mbarrier that nothing ever completes, with
 * the same wait routine the pipelines use but a limit of limit_ns
 * nanoseconds (1e3 .. 1e9) instead of ~1 s.  The wait gives up, sets
 * GPT2_DEVERR_TIMEOUT_BIT in the device error word (read it with
 * gpt2_get_error) and the kernel returns; *gave_up (a DEVICE int) is set
 * to 1 when the wait gave up, 0 if it had completed.  Nothing traps: the
 * device stays usable for the next call.  The pages have no counterpart of
 * this call: it checks the library's own error path.  GPT2_ERR_ARG for a
 * null gave_up or a limit outside the range. */
GPT2_API int gpt2_diag_wait_timeout(long long limit_ns, int* gave_up, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GPT2FWD_H */
