// kernels.cuh -- launchers of the library's kernels (internal interface).
#pragma once

#include "common.cuh"

namespace gpt2 {

constexpr int kMaxDevices = 64;
int num_sms();  // SM count of the current device (cached)

// rowwise.cu
void launch_encoder(float* out, const int* tok, const float* wte, const float* wpe, int N, int T, int C, int V,
                    cudaStream_t s);
void launch_encoder_pos(float* out, const int* tok, const float* wte, const float* wpe, int B, int pos, int C, int V,
                        cudaStream_t s);
void launch_layernorm_f32(float* out, float* mean, float* rstd, const float* inp, const float* w, const float* b,
                          int N, int C, cudaStream_t s);
void launch_layernorm_bf16(__nv_bfloat16* out, const float* inp, const float* w, const float* b, int N, int C,
                           cudaStream_t s);
void launch_gelu(float* out, const float* inp, int n, cudaStream_t s);
void launch_residual(float* out, const float* a, const float* b, int n, cudaStream_t s);
void launch_softmax(float* probs, const float* logits, int N, int V, int Vp, cudaStream_t s);
void launch_argmax(int* next, const float* logits, int B, int V, int Vp, cudaStream_t s);
void launch_f32_to_bf16(__nv_bfloat16* out, const float* in, long long n, cudaStream_t s);
void launch_kv_store_f32(float* cache, const float* qkv, int B, int T, int C, int NH, int maxT, int pos0,
                         cudaStream_t s);
void launch_kv_store_bf16(__nv_bfloat16* cache, const __nv_bfloat16* qkv, int B, int T, int C, int NH, int maxT,
                          int pos0, cudaStream_t s);

// gemm_tc.cu: D[M,N] = A[M,K] B[N,K]^T on tcgen05 tensor cores, A and B
// K-major (row-major [rows, K]), fp32 accumulation in TMEM, fused epilogue.
enum GemmEpilogue {
  kEpiF32 = 0,       // out fp32 = acc (+ bias)
  kEpiBF16 = 1,      // out bf16 = acc (+ bias)
  kEpiGeluBF16 = 2,  // out bf16 = GELU(acc + bias)
  kEpiResidF32 = 3   // out fp32 = out + acc (+ bias), in place
};
// ab_bf16: operands bf16 (kind::f16) when true, fp32 (kind::tf32) when false.
// Returns a GPT2_ERR_* code (tensor-map encoding can fail on bad strides).
int launch_gemm_tc(void* out, const void* A, const void* B, const float* bias, int M, int N, int K, int epi,
                   bool ab_bf16, cudaStream_t s);

// gemm_simt.cu: fp32 CUDA-core GEMM (GPT2_FP32 mode), out = A W^T + bias,
// then optional GELU or residual accumulation (out += ...).
void launch_gemm_simt(float* out, const float* A, const float* W, const float* bias, int M, int N, int K, int epi,
                      cudaStream_t s);

// attention.cu
// bf16 tensor-core causal attention (head size 16, 32 or 64) from a bf16 QKV
// buffer [B,T,3C]; output fp32 or bf16 [B,T,C].
int launch_attention_bf16(void* out, bool out_bf16, const __nv_bfloat16* qkv, int B, int T, int C, int NH,
                           cudaStream_t s);
// fp32 CUDA-core causal attention (head size 16, 32 or 64).
int launch_attention_f32(float* out, const float* qkv, int B, int T, int C, int NH, cudaStream_t s);
// Decode attention: one query per sequence (row b of qkv [B,3C]) against the
// cache positions [0, pos]; output [B,C].
void launch_decode_attention_bf16(void* out, bool out_bf16, const __nv_bfloat16* qkv, const __nv_bfloat16* kcache,
                                  const __nv_bfloat16* vcache, int B, int C, int NH, int maxT, int pos,
                                  float* scratch, cudaStream_t s);
void launch_decode_attention_f32(float* out, const float* qkv, const float* kcache, const float* vcache, int B,
                                 int C, int NH, int maxT, int pos, float* scratch, cudaStream_t s);
size_t decode_attention_scratch_floats(int B, int C, int NH, int maxT);

}  // namespace gpt2
