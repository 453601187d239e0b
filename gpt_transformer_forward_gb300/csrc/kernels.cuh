// kernels.cuh -- launchers of the library's kernels (internal interface).
#pragma once

#include "common.cuh"

namespace gpt2 {

constexpr int kMaxDevices = 64;
int num_sms();  // SM count of the current device (cached)
// Records a CUDA error's text for gpt2_last_cuda_error(), clears it from the
// runtime, and returns GPT2_ERR_CUDA.
int note_cuda_error(cudaError_t e);

// Programmatic dependent launch.  Inside a PdlScope(true) on the calling
// thread (a 16-bit decode step, greedy argmax) the kernels below that call
// pdl_wait() before touching dependent memory are launched with the
// programmatic-stream-serialization attribute, so that each one's launch and
// prologue overlap the tail of the kernel before it.
bool pdl_on();
class PdlScope {
 public:
  explicit PdlScope(bool on);
  ~PdlScope();
  PdlScope(const PdlScope&) = delete;
  PdlScope& operator=(const PdlScope&) = delete;

 private:
  bool prev_;
};

// Launches a kernel whose body begins with pdl_wait() (or waits before its
// first dependent access), with the attribute when pdl_on().
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_on() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Where the cached keys and values of (sequence b, head h, position p) live
// inside one layer's K (or V) half of a KV cache.  Dense (table == nullptr):
// [B][NH][maxT][hs], row (b * NH + h) * maxT + p.  Paged: a pool of blocks
// [num_blocks][NH][2^lbs][hs]; position p of sequence b is in block
// table[b * max_blocks + p / 2^lbs], row (block * NH + h) * 2^lbs + p % 2^lbs.
constexpr int kMaxBlocksPerSeq = 1024;  // block-table entries per sequence (paged layout)
struct KVRows {
  const int* table;
  int lbs;
  int max_blocks;
  int num_blocks;
  int maxT;
  int capacity;  // positions one sequence can hold
};

// rowwise.cu
void launch_encoder(float* out, const int* tok, const float* wte, const float* wpe, int N, int T, int C, int V,
                    cudaStream_t s);
// Decode-step encoder: row b is token tok[b] at position pos (pos_arr[b]
// when pos_arr is given; one outside [0, maxT) is flagged and read as 0).
void launch_encoder_pos(float* out, const int* tok, const float* wte, const float* wpe, int B, int pos,
                        const int* pos_arr, int maxT, int C, int V, cudaStream_t s);
void launch_layernorm_f32(float* out, float* mean, float* rstd, const float* inp, const float* w, const float* b,
                          int N, int C, cudaStream_t s);
// LayerNorm writing the 16-bit operand type T (bf16 or fp16)
template <typename T>
void launch_layernorm_16(T* out, const float* inp, const float* w, const float* b, int N, int C, cudaStream_t s);
// x += y and out = LN(x) in one pass (y and out 16-bit); x is written back
// unless write_x is false
template <typename T16>
void launch_residual_layernorm_16(float* x, const T16* y, T16* out, const float* w, const float* b, int N, int C,
                                  bool write_x, cudaStream_t s);
void launch_gelu(float* out, const float* inp, int n, cudaStream_t s);
void launch_residual(float* out, const float* a, const float* b, int n, cudaStream_t s);
// The type of the probabilities a softmax writes (the values of the C
// ABI's GPT2_PROBS_*): fp32, or the fp32 value rounded to fp16 or bf16.
enum ProbsType { kProbsF32 = 0, kProbsF16 = 1, kProbsBF16 = 2 };
void launch_softmax(void* probs, int probs_type, const float* logits, int N, int V, int Vp, cudaStream_t s);
void launch_argmax(int* next, const float* logits, int B, int V, int Vp, cudaStream_t s);
template <typename T>
void launch_f32_to_16(T* out, const float* in, long long n, cudaStream_t s);
// Copies the keys and values of rows [0, T) of each sequence from the QKV
// buffer [B*T, 3C] into one layer's cache halves kc, vc (positions 0..T-1).
void launch_kv_store_f32(float* kc, float* vc, const float* qkv, int B, int T, int C, int NH, const KVRows& rows,
                         cudaStream_t s);
// 16-bit cache (bf16 or fp16: a plain copy of 2-byte elements)
void launch_kv_store_16(uint16_t* kc, uint16_t* vc, const uint16_t* qkv, int B, int T, int C, int NH,
                        const KVRows& rows, cudaStream_t s);

// Encodes a tiled TMA map with the given shared-memory swizzle: dims[0]
// innermost (in elements), strides_bytes[i] the byte stride of dimension
// i + 1, box the box extent per dimension.  false when the driver rejects
// it.  encode_tensor_map_sw128: the 128-byte swizzle.
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle);
bool encode_tensor_map_sw128(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                             const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box);

// gemm_tc.cu: D[M,N] = A[M,K] B[N,K]^T on tcgen05 tensor cores, A and B
// K-major (row-major [rows, K]), fp32 accumulation in TMEM, fused epilogue.
enum GemmEpilogue {
  kEpiF32 = 0,       // out fp32 = acc (+ bias)
  kEpiOut16 = 1,     // out 16-bit (the operand type) = acc (+ bias)
  kEpiGelu16 = 2,    // out 16-bit = GELU(acc + bias)
  kEpiResidF32 = 3,  // out fp32 = resid + acc (+ bias): resid is out (in place) unless given
  kEpiLogits = 4,    // out fp32 = acc, plus per-(row, 256-column tile) softmax statistics
  kEpiGeluBwdF32 = 5, // out fp32 = acc * GELU'(aux), aux the fp32 [M,N] GELU input (tf32 operands only)
  kEpiGeluDualF32 = 6 // out fp32 = acc (+ bias), and aux fp32 = GELU(out) (tf32 operands only)
};
// Operand types of the tensor-core kernels.
enum OperandType { kOpBF16 = 0, kOpF16 = 1, kOpTF32 = 2 };
// Returns a GPT2_ERR_* code (tensor-map encoding can fail on bad strides).
// The 16-bit epilogues exist for the bf16 and fp16 operand types.  resid:
// a second fp32 [M,N] tensor of the epilogue, M > kSkinnyMaxRows: the
// residual epilogue's addend (out itself, in place, when null),
// kEpiGeluBwdF32's GELU input or kEpiGeluDualF32's GELU output (required).
int launch_gemm_tc(void* out, const void* A, const void* B, const float* bias, int M, int N, int K, int epi, int op,
                   cudaStream_t s, const float* resid = nullptr);

// The same product (fp32 out, no bias) with the K range split over
// concurrently running units when the tiles alone would leave most SMs
// idle (few, long tiles: a weight gradient, K = the tokens): each split's
// fp32 product goes to its slice of `partials` ([splits][M][N], at most
// partial_floats floats), then one kernel sums the slices in order into out
// (deterministic).  Falls back to one launch when splitting does not pay.
int launch_gemm_tc_splitk(float* out, float* partials, size_t partial_floats, const void* A, const void* B, int M,
                          int N, int K, int op, cudaStream_t s);
// the number of K splits that launch chooses
int splitk_choose(int M, int N, int K, int op, size_t partial_floats);

// gemm_skinny.cu: the same product for M <= 64 rows (not the LM-head
// epilogue): weight blocks of 128 rows, K split over the CTAs of a cluster,
// reduced through distributed shared memory.  launch_gemm_tc routes small M
// here.
int launch_gemm_skinny(void* out, const void* A, const void* W, const float* bias, int M, int N, int K, int epi,
                       int op, cudaStream_t s);
constexpr int kSkinnyMaxRows = 64;

// The LM head: logits = A B^T (no bias) and row_stats[row * blocks + i] =
// (max, sum of exp(x - max)) over the columns < V of column block i (128
// columns), blocks = logits_stat_blocks(N) (a block past V holds (-inf, 0)).
int launch_gemm_logits(float* logits, float2* row_stats, const void* A, const void* B, int M, int N, int K, int V,
                       int op, cudaStream_t s);
int logits_stat_blocks(int N);
// Softmax from those statistics: one read of the logits, one write.
void launch_softmax_from_stats(void* probs, int probs_type, const float* logits, const float2* row_stats, int tiles,
                               int N, int V, int Vp, cudaStream_t s);

// gemm_simt.cu: fp32 CUDA-core GEMM (GPT2_FP32 mode), out = A W^T + bias,
// then optional GELU or residual accumulation (out += ...).
void launch_gemm_simt(float* out, const float* A, const float* W, const float* bias, int M, int N, int K, int epi,
                      cudaStream_t s);

// attention.cu
// Tensor-core causal attention (head size 16, 32 or 64) from a 16-bit QKV
// buffer [B,T,3C] of operand type op (kOpBF16 or kOpF16); output fp32, or
// the operand type when out16.
int launch_attention_16(void* out, bool out16, const void* qkv, int op, int B, int T, int C, int NH,
                        cudaStream_t s);
// The same on tcgen05/TMEM (attention_tc.cu), head size 64 only; lse
// (optional): [B][NH][attn_bwd_padded_len(T)] floats, each row's
// log-sum-exp of the scaled scores in log2 units (m + log2 l).
int launch_attention_tc05(void* out, bool out16, const void* qkv, int op, int B, int T, int C, int NH,
                          cudaStream_t s, float* lse = nullptr);
// fp32 CUDA-core causal attention (head size 16, 32 or 64).
int launch_attention_f32(float* out, const float* qkv, int B, int T, int C, int NH, cudaStream_t s);
// Decode attention: one query per sequence (row b of qkv [B,3C]) against the
// cache positions [0, pos] (pos_arr[b] when pos_arr is given), the key and
// value of position pos taken from qkv and appended to the cache; output
// [B,C].  kcache, vcache: the layer's K and V halves, laid out as `rows`.
void launch_decode_attention_16(void* out, bool out16, const void* qkv, void* kcache, void* vcache, int op, int B,
                                int C, int NH, int pos, const int* pos_arr, const KVRows& rows, cudaStream_t s);
void launch_decode_attention_f32(float* out, const float* qkv, float* kcache, float* vcache, int B, int C, int NH,
                                 int pos, const int* pos_arr, const KVRows& rows, cudaStream_t s);

// attention_bwd.cu: the backward of causal attention in fp32; Lrow, Drow:
// [B][NH][T] floats of scratch (the forward's row statistic, rowsum dO*O).
int launch_attention_backward(float* dqkv, const float* dout, const float* qkv, const float* out, float* Lrow,
                              float* Drow, int B, int T, int C, int NH, cudaStream_t s);

// attention_bwd_tc.cu: the backward of causal attention on tcgen05, head
// size 64, bf16 operands.  attn_bwd_padded_len(T): T rounded up to 128, the
// row length of the [B][NH][Tp] statistics.  launch_attn_bwd_prep: dO16
// [B,T,C] bf16 = dout, Dv = rowsum(dout * out) per head, Dv and Lse zero
// past T.  launch_attention_backward_tc05: dqkv [B,T,3C] fp32 (every
// element written) from qkv16 [B,T,3C] and do16 [B,T,C] bf16, Lse from the
// forward (launch_attention_tc05) and Dv.
int attn_bwd_padded_len(int T);
void launch_attn_bwd_prep(void* do16, float* Dv, float* Lse, const float* dout, const float* out, int B, int T, int C,
                          int NH, cudaStream_t s);
int launch_attention_backward_tc05(float* dqkv, const void* qkv16, const void* do16, const float* Lse,
                                   const float* Dv, int B, int T, int C, int NH, cudaStream_t s);

// train.cu: the training step's kernels (fp32).  column_parts(rows): the
// partial sums a column reduction over `rows` rows keeps in scratch.
int column_parts(int rows);
void launch_transpose(float* out, const float* in, int rows, int cols, cudaStream_t s);
// softmax cross-entropy over the first V of Vp columns: losses[n], the mean
// into loss[0], dlogits (p - onehot) / N written over the logits
void launch_crossentropy(float* logits, float* losses, float* loss, const int* targets, int N, int V, int Vp,
                         cudaStream_t s);
// out[c] (+)= sum over rows of in[r][c]; part: column_parts(rows) x cols floats
void launch_column_sum(float* out, float* part, const float* in, int rows, int cols, bool accumulate, cudaStream_t s);
// dx (+)= LayerNorm backward; dw, db set; part: 2 x column_parts(N) x C floats
void launch_layernorm_backward(float* dx, float* dw, float* db, float* part, const float* dy, const float* x,
                               const float* w, const float* mean, const float* rstd, int N, int C, bool accumulate,
                               cudaStream_t s);
void launch_gelu_backward(float* dinp, const float* inp, const float* dout, long long n, cudaStream_t s);
// dwpe rows [0, T) set; dwte[tok] += dx
void launch_encoder_backward(float* dwte, float* dwpe, const float* dx, const int* tok, int B, int T, int C, int V,
                             cudaStream_t s);
void launch_adamw(float* p, const float* g, float* m, float* v, long long n, float lr, float b1, float b2, float eps,
                  float wd, int t, cudaStream_t s);

}  // namespace gpt2
