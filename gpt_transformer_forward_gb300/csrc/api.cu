// api.cu -- the C ABI (declared in include/gpt2fwd.h): argument checks,
// workspace and weight-packing layouts, and the orchestration of the
// forward pass and of the decode step on the caller's stream.
//
// Forward pass order (pre-LayerNorm GPT-2 blocks; the ECE408 GPT-2 project
// page names the kernels, llm.c's profile splits the step into encoder,
// forward blocks and classifier):
//   encoder -> L x [LN1 -> QKV GEMM(+bias) -> attention -> attn-proj GEMM
//   (+bias, +residual in place) -> LN2 -> FC GEMM(+bias, GELU) -> FC-proj
//   GEMM(+bias, +residual in place)] -> LN_f -> LM-head GEMM (tied wte) ->
//   softmax.
// In the 16-bit modes (GPT2_BF16, GPT2_FP16) LayerNorm, the QKV and GELU
// epilogues and attention write the 16-bit operand type directly, because
// that is the only form in which the next tensor-core step consumes them;
// the residual stream x, the logits and the probabilities stay fp32.
#include <stdio.h>

#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "kernels.cuh"

namespace gpt2 {

int num_sms() {
  static int cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

namespace {
thread_local std::string g_last_cuda_error;
}  // namespace

namespace {
thread_local bool t_pdl = false;
}
bool pdl_on() { return t_pdl; }
PdlScope::PdlScope(bool on) : prev_(t_pdl) { t_pdl = on; }
PdlScope::~PdlScope() { t_pdl = prev_; }

int note_cuda_error(cudaError_t e) {
  g_last_cuda_error = cudaGetErrorString(e);
  cudaGetLastError();
  return GPT2_ERR_CUDA;
}

namespace {

int check_launch() {
  const cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess) {
    g_last_cuda_error = cudaGetErrorString(e);
    cudaGetLastError();
    return GPT2_ERR_CUDA;
  }
  return GPT2_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

#define RETURN_IF(cond, code) \
  do {                        \
    if (cond) return (code);  \
  } while (0)

#define TRY(expr)                   \
  do {                              \
    const int _rc = (expr);         \
    if (_rc != GPT2_OK) return _rc; \
  } while (0)

bool valid_precision(int p) { return p == GPT2_FP32 || p == GPT2_TF32 || p == GPT2_BF16 || p == GPT2_FP16; }
// 16-bit operand modes keep GEMM operands, attention inputs and the KV cache in
// the 16-bit type; the tensor-core operand type of each mode:
bool is16(int p) { return p == GPT2_BF16 || p == GPT2_FP16; }
int op_of(int p) { return p == GPT2_FP16 ? kOpF16 : (p == GPT2_TF32 ? kOpTF32 : kOpBF16); }

// fp32 -> the 16-bit operand type of a 16-bit precision mode
void to16(int precision, void* out, const float* in, long long n, cudaStream_t s) {
  if (precision == GPT2_FP16)
    launch_f32_to_16(static_cast<__half*>(out), in, n, s);
  else
    launch_f32_to_16(static_cast<__nv_bfloat16*>(out), in, n, s);
}

int check_config(const GPT2Config* c) {
  RETURN_IF(c == nullptr, GPT2_ERR_ARG);
  RETURN_IF(c->max_seq_len <= 0 || c->vocab_size <= 0 || c->padded_vocab_size < c->vocab_size ||
                c->num_layers <= 0 || c->num_heads <= 0 || c->channels <= 0,
            GPT2_ERR_ARG);
  RETURN_IF(c->channels % c->num_heads != 0, GPT2_ERR_SHAPE);
  RETURN_IF(c->channels % 8 != 0 || c->padded_vocab_size % 4 != 0, GPT2_ERR_SHAPE);
  return GPT2_OK;
}

// every attention kernel (tensor-core, fp32 and decode) handles head sizes 16, 32, 64
int check_attention_shape(int C, int NH) {
  const int hs = C / NH;
  return (hs == 16 || hs == 32 || hs == 64) ? GPT2_OK : GPT2_ERR_UNSUPPORTED;
}

// ------------------------------------------------ parameter tensor offsets
struct ParamOffsets {
  size_t wte, wpe, ln1w, ln1b, qkvw, qkvb, attprojw, attprojb, ln2w, ln2b, fcw, fcb, fcprojw, fcprojb, lnfw, lnfb,
      total;
};

ParamOffsets param_offsets(const GPT2Config* c) {
  const size_t C = c->channels, L = c->num_layers, Vp = c->padded_vocab_size, maxT = c->max_seq_len;
  ParamOffsets o;
  size_t p = 0;
  o.wte = p; p += Vp * C;
  o.wpe = p; p += maxT * C;
  o.ln1w = p; p += L * C;
  o.ln1b = p; p += L * C;
  o.qkvw = p; p += L * 3 * C * C;
  o.qkvb = p; p += L * 3 * C;
  o.attprojw = p; p += L * C * C;
  o.attprojb = p; p += L * C;
  o.ln2w = p; p += L * C;
  o.ln2b = p; p += L * C;
  o.fcw = p; p += L * 4 * C * C;
  o.fcb = p; p += L * 4 * C;
  o.fcprojw = p; p += L * 4 * C * C;
  o.fcprojb = p; p += L * C;
  o.lnfw = p; p += C;
  o.lnfb = p; p += C;
  o.total = p;
  return o;
}

// bf16 copies of the five weight matrices, each 256-byte aligned
struct PackedOffsets {
  size_t wte, qkvw, attprojw, fcw, fcprojw, total;  // byte offsets
};

PackedOffsets packed_offsets(const GPT2Config* c) {
  const size_t C = c->channels, L = c->num_layers, Vp = c->padded_vocab_size;
  PackedOffsets o;
  size_t p = 0;
  o.wte = p; p = round_up(p + Vp * C * 2, 256);
  o.qkvw = p; p = round_up(p + L * 3 * C * C * 2, 256);
  o.attprojw = p; p = round_up(p + L * C * C * 2, 256);
  o.fcw = p; p = round_up(p + L * 4 * C * C * 2, 256);
  o.fcprojw = p; p = round_up(p + L * 4 * C * C * 2, 256);
  o.total = p;
  return o;
}

// ---------------------------------------------------------- workspace
struct Workspace {
  size_t x, ln, qkv, qkv16, att, fch, stats, total;  // byte offsets
};

Workspace workspace_layout(const GPT2Config* c, int B, int T, int precision) {
  const size_t N = static_cast<size_t>(B) * T, C = c->channels;
  const size_t act = is16(precision) ? 2 : 4;  // operand buffers
  Workspace w;
  size_t p = 0;
  w.x = p; p = round_up(p + N * C * 4, 256);
  w.ln = p; p = round_up(p + N * C * act, 256);
  w.qkv = p; p = round_up(p + N * 3 * C * act, 256);
  w.qkv16 = p;
  if (precision == GPT2_TF32) p = round_up(p + N * 3 * C * 2, 256);  // bf16 copy for the attention kernel
  w.att = p; p = round_up(p + N * C * act, 256);
  w.fch = p; p = round_up(p + N * 4 * C * act, 256);
  w.stats = p; p = round_up(p + N * logits_stat_blocks(c->padded_vocab_size) * sizeof(float2), 256);  // softmax statistics
  w.total = p;
  return w;
}

size_t kv_elem_bytes(int precision) { return is16(precision) ? 2 : 4; }

// elements of one layer's cache slab [2][B][NH][maxT][hs]
size_t kv_layer_elems(const GPT2Config* c, int B) {
  return 2ull * B * c->num_heads * c->max_seq_len * (c->channels / c->num_heads);
}

// elements of one layer's slab of a paged pool [2][num_blocks][NH][block][hs]
size_t paged_layer_elems(const GPT2Config* c, int num_blocks, int block_size) {
  return 2ull * num_blocks * c->num_heads * block_size * (c->channels / c->num_heads);
}

// A KV cache as the forward pass and the decode step address it: the base
// of layer 0's slab, the row layout inside one K or V half, and the
// elements of a layer's slab (its K half, then its V half).
struct KVLayout {
  void* base;
  KVRows rows;
  size_t layer_elems;
};

KVLayout dense_kv(const GPT2Config* c, void* cache, int B) {
  KVLayout k;
  k.base = cache;
  k.rows = KVRows{nullptr, 0, 1, B, c->max_seq_len, c->max_seq_len};
  k.layer_elems = kv_layer_elems(c, B);
  return k;
}

int log2_exact(int v) {  // -1 unless v is a power of two
  if (v <= 0 || (v & (v - 1)) != 0) return -1;
  int l = 0;
  while ((1 << l) < v) ++l;
  return l;
}

// Checks a caller's paged cache description on the host and builds its
// layout; positions [0, T) must fit one sequence's blocks when T > 0.
int paged_kv(const GPT2Config* c, const GPT2PagedKVCache* p, int T, KVLayout* out) {
  RETURN_IF(p == nullptr || p->pool == nullptr || p->block_table == nullptr, GPT2_ERR_ARG);
  const int lbs = log2_exact(p->block_size);
  RETURN_IF(lbs < 0 || p->num_blocks <= 0 || p->max_blocks_per_seq <= 0, GPT2_ERR_ARG);
  RETURN_IF(p->max_blocks_per_seq > kMaxBlocksPerSeq, GPT2_ERR_SHAPE);
  RETURN_IF((reinterpret_cast<uintptr_t>(p->pool) & 15u) != 0 ||
                (reinterpret_cast<uintptr_t>(p->block_table) & 3u) != 0,
            GPT2_ERR_ALIGN);
  const long long cap = std::min<long long>(c->max_seq_len, static_cast<long long>(p->max_blocks_per_seq) << lbs);
  RETURN_IF(T > cap, GPT2_ERR_SHAPE);
  out->base = p->pool;
  out->rows = KVRows{p->block_table, lbs, p->max_blocks_per_seq, p->num_blocks, c->max_seq_len, static_cast<int>(cap)};
  out->layer_elems = paged_layer_elems(c, p->num_blocks, p->block_size);
  return GPT2_OK;
}

// One GEMM site: picks the kernel for the precision mode.
int gemm(int precision, void* out, const void* A, const void* W, const float* bias, int M, int N, int K, int epi,
         cudaStream_t s) {
  if (precision == GPT2_FP32) {
    launch_gemm_simt(static_cast<float*>(out), static_cast<const float*>(A), static_cast<const float*>(W), bias, M,
                     N, K, epi, s);
    return check_launch();
  }
  if (precision == GPT2_TF32 && epi == kEpiGelu16) {
    // tf32 operands with an fp32 GELU output: GEMM then the GELU kernel
    TRY(launch_gemm_tc(out, A, W, bias, M, N, K, kEpiF32, kOpTF32, s));
    launch_gelu(static_cast<float*>(out), static_cast<const float*>(out), M * N, s);
    return check_launch();
  }
  return launch_gemm_tc(out, A, W, bias, M, N, K, epi, op_of(precision), s);
}

// Records a CUDA event on the stream after each stage of the forward pass;
// stage_ms[k] accumulates the time between the event before and after each
// occurrence of stage k.
struct StageProfiler {
  cudaStream_t stream;
  std::vector<cudaEvent_t> events;
  std::vector<int> stages;  // stage of the interval ending at events[i + 1]
  int begin() {
    return record(-1);
  }
  int record(int stage) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return GPT2_ERR_CUDA;
    events.push_back(e);
    if (stage >= 0) stages.push_back(stage);
    return cudaEventRecord(e, stream) == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
  }
  int finish(float* stage_ms, int n_stages) {
    int rc = cudaEventSynchronize(events.back()) == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
    for (size_t i = 0; rc == GPT2_OK && i + 1 < events.size(); ++i) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, events[i], events[i + 1]) != cudaSuccess) rc = GPT2_ERR_CUDA;
      if (stages[i] < n_stages) stage_ms[stages[i]] += ms;
    }
    for (cudaEvent_t e : events) cudaEventDestroy(e);
    events.clear();
    return rc;
  }
};

// ----------------------------------------------------- training workspace
// fp32 activations of every layer kept for the backward, and the backward's
// scratch; offsets in bytes, each 256-byte aligned.
struct TrainLayout {
  size_t xin, xmid, ln1, ln2, ln1m, ln1r, ln2m, ln2r, qkv, qkv16, att, fc, fcg, lnf, lnfm, lnfr, logits, losses, dx,
      dh, dt, dt2, dqkv, tA, tB, Wt, part, attn, lse, splitk, total;
};

// the K-split partial products of the weight gradients: up to 16 slices of
// the largest one (4C x C)
size_t kSplitkFloats(size_t C) { return 16 * 4 * C * C; }

TrainLayout train_layout(const GPT2Config* c, int B, int T) {
  const size_t N = static_cast<size_t>(B) * T, C = c->channels, L = c->num_layers, Vp = c->padded_vocab_size;
  const size_t NC = N * C, F = sizeof(float);
  const size_t wide = Vp > 4 * C ? Vp : 4 * C;
  TrainLayout t;
  size_t p = 0;
  auto take = [&](size_t floats) {
    const size_t at = p;
    p = round_up(p + floats * F, 256);
    return at;
  };
  t.xin = take((L + 1) * NC);
  t.xmid = take(L * NC);
  t.ln1 = take(L * NC);
  t.ln2 = take(L * NC);
  t.ln1m = take(L * N);
  t.ln1r = take(L * N);
  t.ln2m = take(L * N);
  t.ln2r = take(L * N);
  t.qkv = take(L * 3 * NC);
  t.qkv16 = take((L * 3 * NC + 1) / 2);  // every layer's bf16 copy of qkv (the tf32 mode's attention operands)
  t.att = take(L * NC);
  t.fc = take(L * 4 * NC);
  t.fcg = take(L * 4 * NC);
  t.lnf = take(NC);
  t.lnfm = take(N);
  t.lnfr = take(N);
  t.logits = take(N * Vp);
  t.losses = take(N);
  t.dx = take(NC);
  t.dh = take(NC);
  t.dt = take(4 * NC);
  t.dt2 = take(4 * NC);
  t.dqkv = take(3 * NC);
  t.tA = take(N * wide);
  t.tB = take(4 * NC);
  t.Wt = take(wide * C);
  t.part = take(2 * static_cast<size_t>(column_parts(static_cast<int>(N))) * wide);
  t.attn = take(2 * static_cast<size_t>(B) * c->num_heads * attn_bwd_padded_len(T));
  t.lse = take(L * static_cast<size_t>(B) * c->num_heads * attn_bwd_padded_len(T));
  t.splitk = take(kSplitkFloats(C));
  t.total = p;
  return t;
}

}  // namespace
}  // namespace gpt2

using namespace gpt2;

// ====================================================================== ABI
extern "C" {

int encoder_forward(float* out, const int* tok, const float* wte, const float* wpe, int B, int T, int C, int V,
                    void* stream) {
  RETURN_IF(!out || !tok || !wte || !wpe, GPT2_ERR_ARG);
  RETURN_IF(B < 0 || T < 0 || C <= 0 || V <= 0, GPT2_ERR_ARG);
  RETURN_IF(C % 4 != 0, GPT2_ERR_SHAPE);
  RETURN_IF(!aligned16(out) || !aligned16(wte) || !aligned16(wpe), GPT2_ERR_ALIGN);
  if (B == 0 || T == 0) return GPT2_OK;
  launch_encoder(out, tok, wte, wpe, B * T, T, C, V, as_stream(stream));
  return check_launch();
}

int layernorm_forward(float* out, float* mean, float* rstd, const float* inp, const float* w, const float* b, int N,
                      int C, void* stream) {
  RETURN_IF(!out || !inp || !w || !b, GPT2_ERR_ARG);
  RETURN_IF(N < 0 || C <= 0, GPT2_ERR_ARG);
  RETURN_IF(C % 4 != 0, GPT2_ERR_SHAPE);
  RETURN_IF(!aligned16(out) || !aligned16(inp) || !aligned16(w) || !aligned16(b), GPT2_ERR_ALIGN);
  if (N == 0) return GPT2_OK;
  launch_layernorm_f32(out, mean, rstd, inp, w, b, N, C, as_stream(stream));
  return check_launch();
}

size_t matmul_workspace_size(int N, int C, int OC, int precision) {
  if (!is16(precision) || N <= 0 || C <= 0 || OC <= 0) return 0;
  return round_up(static_cast<size_t>(N) * C * 2, 256) + round_up(static_cast<size_t>(OC) * C * 2, 256);
}

int matmul_forward(float* out, const float* inp, const float* W, const float* bias, int N, int C, int OC,
                   int precision, void* workspace, size_t ws_bytes, void* stream) {
  RETURN_IF(!out || !inp || !W, GPT2_ERR_ARG);
  RETURN_IF(N < 0 || C <= 0 || OC <= 0 || !valid_precision(precision), GPT2_ERR_ARG);
  RETURN_IF(!aligned16(out) || !aligned16(inp) || !aligned16(W) || (bias && !aligned16(bias)), GPT2_ERR_ALIGN);
  if (N == 0) return GPT2_OK;
  cudaStream_t s = as_stream(stream);
  if (precision == GPT2_FP32) return gemm(precision, out, inp, W, bias, N, OC, C, kEpiF32, s);
  RETURN_IF(C % 8 != 0 || OC % 4 != 0, GPT2_ERR_SHAPE);
  if (precision == GPT2_TF32) return launch_gemm_tc(out, inp, W, bias, N, OC, C, kEpiF32, kOpTF32, s);
  const size_t need = matmul_workspace_size(N, C, OC, precision);
  RETURN_IF(workspace == nullptr || ws_bytes < need, GPT2_ERR_WORKSPACE);
  RETURN_IF((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0, GPT2_ERR_ALIGN);
  void* a16 = workspace;
  void* w16 = static_cast<uint8_t*>(workspace) + round_up(static_cast<size_t>(N) * C * 2, 256);
  to16(precision, a16, inp, static_cast<long long>(N) * C, s);
  to16(precision, w16, W, static_cast<long long>(OC) * C, s);
  TRY(check_launch());
  return launch_gemm_tc(out, a16, w16, bias, N, OC, C, kEpiF32, op_of(precision), s);
}

size_t attention_workspace_size(int B, int T, int C, int precision) {
  if (precision == GPT2_FP32 || B <= 0 || T <= 0 || C <= 0) return 0;
  return round_up(static_cast<size_t>(B) * T * 3 * C * 2, 256);
}

int attention_forward(float* out, const float* qkv, int B, int T, int C, int NH, int precision, void* workspace,
                      size_t ws_bytes, void* stream) {
  RETURN_IF(!out || !qkv, GPT2_ERR_ARG);
  RETURN_IF(B < 0 || T < 0 || C <= 0 || NH <= 0 || !valid_precision(precision), GPT2_ERR_ARG);
  RETURN_IF(C % NH != 0, GPT2_ERR_SHAPE);
  TRY(check_attention_shape(C, NH));
  RETURN_IF(!aligned16(out) || !aligned16(qkv), GPT2_ERR_ALIGN);
  if (B == 0 || T == 0) return GPT2_OK;
  cudaStream_t s = as_stream(stream);
  if (precision == GPT2_FP32) {
    TRY(launch_attention_f32(out, qkv, B, T, C, NH, s));
    return check_launch();
  }
  RETURN_IF(workspace == nullptr || ws_bytes < attention_workspace_size(B, T, C, precision), GPT2_ERR_WORKSPACE);
  RETURN_IF(!aligned16(workspace), GPT2_ERR_ALIGN);
  // GPT2_TF32 runs the bf16 kernel; GPT2_BF16 / GPT2_FP16 their own type
  const int p16 = precision == GPT2_FP16 ? GPT2_FP16 : GPT2_BF16;
  to16(p16, workspace, qkv, static_cast<long long>(B) * T * 3 * C, s);
  TRY(launch_attention_16(out, false, workspace, op_of(p16), B, T, C, NH, s));
  return check_launch();
}

// the 16-bit backward's workspace: bf16 copies of qkv and dout, the bf16
// output of the forward recompute that yields the row statistic, then the
// statistic L and rowsum(dout * out), [B][NH][Tp] each
struct AttnBwd16Layout {
  size_t qkv16, do16, o16, lse, dvec, total;
};
AttnBwd16Layout attn_bwd16_layout(int B, int T, int C, int NH) {
  const size_t N = static_cast<size_t>(B) * T, S = static_cast<size_t>(B) * NH * attn_bwd_padded_len(T);
  AttnBwd16Layout l;
  l.qkv16 = 0;
  l.do16 = l.qkv16 + round_up(N * 3 * C * 2, 256);
  l.o16 = l.do16 + round_up(N * C * 2, 256);
  l.lse = l.o16 + round_up(N * C * 2, 256);
  l.dvec = l.lse + round_up(S * sizeof(float), 256);
  l.total = l.dvec + round_up(S * sizeof(float), 256);
  return l;
}

size_t attention_backward_workspace_size(int B, int T, int C, int NH, int precision) {
  if (B <= 0 || T <= 0 || C <= 0 || NH <= 0 || C % NH != 0) return 0;
  if (precision == GPT2_FP32) return 2 * round_up(static_cast<size_t>(B) * NH * T * sizeof(float), 256);
  if ((precision == GPT2_TF32 || precision == GPT2_BF16) && C / NH == 64) return attn_bwd16_layout(B, T, C, NH).total;
  return 0;
}

int attention_backward(float* dqkv, const float* dout, const float* qkv, const float* out, int B, int T, int C, int NH,
                       int precision, void* workspace, size_t ws_bytes, void* stream) {
  RETURN_IF(!dqkv || !dout || !qkv || !out, GPT2_ERR_ARG);
  RETURN_IF(B < 0 || T < 0 || C <= 0 || NH <= 0 || !valid_precision(precision), GPT2_ERR_ARG);
  RETURN_IF(C % NH != 0, GPT2_ERR_SHAPE);
  TRY(check_attention_shape(C, NH));
  // the 16-bit path: bf16 operands (the gradients need bf16's exponent
  // range), head size 64
  RETURN_IF(precision == GPT2_FP16 || (precision != GPT2_FP32 && C / NH != 64), GPT2_ERR_UNSUPPORTED);
  if (B == 0 || T == 0) return GPT2_OK;
  RETURN_IF(workspace == nullptr || ws_bytes < attention_backward_workspace_size(B, T, C, NH, precision),
            GPT2_ERR_WORKSPACE);
  RETURN_IF(!aligned16(dqkv) || !aligned16(dout) || !aligned16(qkv) || !aligned16(out) || !aligned16(workspace),
            GPT2_ERR_ALIGN);
  cudaStream_t s = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (precision == GPT2_FP32) {
    float* Lrow = reinterpret_cast<float*>(ws);
    float* Drow = reinterpret_cast<float*>(ws + round_up(static_cast<size_t>(B) * NH * T * sizeof(float), 256));
    TRY(launch_attention_backward(dqkv, dout, qkv, out, Lrow, Drow, B, T, C, NH, s));
    return check_launch();
  }
  const AttnBwd16Layout l = attn_bwd16_layout(B, T, C, NH);
  float* lse = reinterpret_cast<float*>(ws + l.lse);
  float* dvec = reinterpret_cast<float*>(ws + l.dvec);
  to16(GPT2_BF16, ws + l.qkv16, qkv, static_cast<long long>(B) * T * 3 * C, s);
  // the forward again, for each row's log-sum-exp (its output is not used)
  TRY(launch_attention_tc05(ws + l.o16, true, ws + l.qkv16, kOpBF16, B, T, C, NH, s, lse));
  launch_attn_bwd_prep(ws + l.do16, dvec, lse, dout, out, B, T, C, NH, s);
  TRY(launch_attention_backward_tc05(dqkv, ws + l.qkv16, ws + l.do16, lse, dvec, B, T, C, NH, s));
  return check_launch();
}

int gelu_forward(float* out, const float* inp, int n, void* stream) {
  RETURN_IF(!out || !inp || n < 0, GPT2_ERR_ARG);
  RETURN_IF(!aligned16(out) || !aligned16(inp), GPT2_ERR_ALIGN);
  if (n == 0) return GPT2_OK;
  launch_gelu(out, inp, n, as_stream(stream));
  return check_launch();
}

int residual_forward(float* out, const float* a, const float* b, int n, void* stream) {
  RETURN_IF(!out || !a || !b || n < 0, GPT2_ERR_ARG);
  RETURN_IF(!aligned16(out) || !aligned16(a) || !aligned16(b), GPT2_ERR_ALIGN);
  if (n == 0) return GPT2_OK;
  launch_residual(out, a, b, n, as_stream(stream));
  return check_launch();
}

static bool valid_probs_type(int t) { return t == GPT2_PROBS_F32 || t == GPT2_PROBS_F16 || t == GPT2_PROBS_BF16; }

int softmax_forward_ex(void* probs, int probs_type, const float* logits, int N, int V, int Vp, void* stream) {
  RETURN_IF(!probs || !logits || N < 0 || V <= 0 || Vp < V || !valid_probs_type(probs_type), GPT2_ERR_ARG);
  RETURN_IF(Vp % 4 != 0, GPT2_ERR_SHAPE);
  RETURN_IF(!aligned16(probs) || !aligned16(logits), GPT2_ERR_ALIGN);
  if (N == 0) return GPT2_OK;
  launch_softmax(probs, probs_type, logits, N, V, Vp, as_stream(stream));
  return check_launch();
}

int softmax_forward(float* probs, const float* logits, int N, int V, int Vp, void* stream) {
  return softmax_forward_ex(probs, GPT2_PROBS_F32, logits, N, V, Vp, stream);
}

int gpt2_argmax(int* next, const float* logits, int B, int V, int Vp, void* stream) {
  RETURN_IF(!next || !logits || B < 0 || V <= 0 || Vp < V, GPT2_ERR_ARG);
  if (B == 0) return GPT2_OK;
  PdlScope pdl(true);  // the argmax kernel waits for its predecessor itself
  launch_argmax(next, logits, B, V, Vp, as_stream(stream));
  return check_launch();
}

size_t gpt2_num_parameters(const GPT2Config* cfg) {
  if (check_config(cfg) != GPT2_OK) return 0;
  return param_offsets(cfg).total;
}

size_t gpt2_packed_weights_size(const GPT2Config* cfg, int precision) {
  if (check_config(cfg) != GPT2_OK || !is16(precision)) return 0;
  return packed_offsets(cfg).total;
}

int gpt2_prepare_weights(const GPT2Config* cfg, const float* params, void* packed, size_t bytes, int precision,
                         void* stream) {
  TRY(check_config(cfg));
  RETURN_IF(!params || !valid_precision(precision), GPT2_ERR_ARG);
  if (!is16(precision)) return GPT2_OK;
  RETURN_IF(!packed, GPT2_ERR_ARG);
  RETURN_IF(bytes < gpt2_packed_weights_size(cfg, precision), GPT2_ERR_WORKSPACE);
  RETURN_IF(!aligned16(params) || (reinterpret_cast<uintptr_t>(packed) & 255u) != 0, GPT2_ERR_ALIGN);
  const ParamOffsets po = param_offsets(cfg);
  const PackedOffsets ko = packed_offsets(cfg);
  const size_t C = cfg->channels, L = cfg->num_layers, Vp = cfg->padded_vocab_size;
  uint8_t* base = static_cast<uint8_t*>(packed);
  cudaStream_t s = as_stream(stream);
  auto conv = [&](size_t dst_off, size_t src_off, size_t n) {
    to16(precision, base + dst_off, params + src_off, static_cast<long long>(n), s);
  };
  conv(ko.wte, po.wte, Vp * C);
  conv(ko.qkvw, po.qkvw, L * 3 * C * C);
  conv(ko.attprojw, po.attprojw, L * C * C);
  conv(ko.fcw, po.fcw, L * 4 * C * C);
  conv(ko.fcprojw, po.fcprojw, L * 4 * C * C);
  return check_launch();
}

size_t gpt2_workspace_size(const GPT2Config* cfg, int B, int T, int precision) {
  if (check_config(cfg) != GPT2_OK || B <= 0 || T <= 0 || !valid_precision(precision)) return 0;
  return workspace_layout(cfg, B, T, precision).total;
}

size_t gpt2_kvcache_size(const GPT2Config* cfg, int B, int precision) {
  if (check_config(cfg) != GPT2_OK || B <= 0 || !valid_precision(precision)) return 0;
  return static_cast<size_t>(cfg->num_layers) * kv_layer_elems(cfg, B) * kv_elem_bytes(precision);
}

// The body shared by the full forward pass and the decode step.  decode
// false: rows are B sequences x T tokens at positions 0..T-1 (their keys and
// values written into kv when it is given: a prefill); decode true: rows are
// the B sequences' tokens at position decode_pos, or pos_arr[b] when pos_arr
// is given (T == 1), attending over and appending to kv.
static int run_forward(const GPT2Config* cfg, const float* params, const void* packed, const int* tok, int B, int T,
                       bool decode, int decode_pos, const int* pos_arr, float* logits, void* probs,
                       const KVLayout* kv, void* workspace, size_t ws_bytes, int precision, cudaStream_t s,
                       StageProfiler* prof = nullptr, int probs_type = GPT2_PROBS_F32) {
  auto mark = [&](int stage) { return prof ? prof->record(stage) : GPT2_OK; };
  const int C = cfg->channels, L = cfg->num_layers, NH = cfg->num_heads, V = cfg->vocab_size;
  const int Vp = cfg->padded_vocab_size, maxT = cfg->max_seq_len;
  const int N = B * T;
  const ParamOffsets po = param_offsets(cfg);
  const Workspace wl = workspace_layout(cfg, B, T, precision);
  RETURN_IF(ws_bytes < wl.total, GPT2_ERR_WORKSPACE);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* x = reinterpret_cast<float*>(ws + wl.x);
  void* ln = ws + wl.ln;
  void* qkv = ws + wl.qkv;
  void* att = ws + wl.att;
  void* fch = ws + wl.fch;
  const bool bf16 = is16(precision);  // 16-bit operand buffers (bf16 or fp16)
  const int op = op_of(precision);
  const PackedOffsets ko = packed_offsets(cfg);
  const uint8_t* pk = static_cast<const uint8_t*>(packed);
  const size_t kv_slab = kv != nullptr ? kv->layer_elems : 0;
  const size_t kv_half = kv_slab / 2;

  // weight matrix of a GEMM site for layer l
  auto wmat = [&](size_t f32_off, size_t bf16_off, size_t per_layer, int l) -> const void* {
    if (bf16) return pk + bf16_off + static_cast<size_t>(l) * per_layer * 2;
    return params + f32_off + static_cast<size_t>(l) * per_layer;
  };
  auto layernorm = [&](void* out, const float* in, size_t w_off, size_t b_off) {
    if (precision == GPT2_FP16)
      launch_layernorm_16(static_cast<__half*>(out), in, params + w_off, params + b_off, N, C, s);
    else if (precision == GPT2_BF16)
      launch_layernorm_16(static_cast<__nv_bfloat16*>(out), in, params + w_off, params + b_off, N, C, s);
    else
      launch_layernorm_f32(static_cast<float*>(out), nullptr, nullptr, in, params + w_off, params + b_off, N, C, s);
  };
  // In the 16-bit modes the attention and MLP projections write their
  // output y (bias added) as 16-bit into the QKV buffer, which is free by
  // then, and the residual add x += y runs in the LayerNorm that reads x
  // next: the same bytes as a residual-accumulating GEMM epilogue plus a
  // plain LayerNorm, without the epilogue's serial read of x.
  void* y16 = qkv;
  auto resid_layernorm = [&](size_t w_off, size_t b_off, bool write_x) {
    if (precision == GPT2_FP16)
      launch_residual_layernorm_16(x, static_cast<const __half*>(y16), static_cast<__half*>(ln), params + w_off,
                                   params + b_off, N, C, write_x, s);
    else
      launch_residual_layernorm_16(x, static_cast<const __nv_bfloat16*>(y16), static_cast<__nv_bfloat16*>(ln),
                                   params + w_off, params + b_off, N, C, write_x, s);
  };

  if (!decode)
    launch_encoder(x, tok, params + po.wte, params + po.wpe, N, T, C, V, s);
  else
    launch_encoder_pos(x, tok, params + po.wte, params + po.wpe, B, decode_pos, pos_arr, maxT, C, V, s);
  TRY(check_launch());
  TRY(mark(GPT2_STAGE_ENCODER));

  for (int l = 0; l < L; ++l) {
    const size_t CC = static_cast<size_t>(C) * C;
    if (bf16 && l > 0)  // the previous layer's MLP output is still to be added
      resid_layernorm(po.ln1w + static_cast<size_t>(l) * C, po.ln1b + static_cast<size_t>(l) * C, true);
    else
      layernorm(ln, x, po.ln1w + static_cast<size_t>(l) * C, po.ln1b + static_cast<size_t>(l) * C);
    TRY(mark(GPT2_STAGE_LN1));
    TRY(gemm(precision, qkv, ln, wmat(po.qkvw, ko.qkvw, 3 * CC, l), params + po.qkvb + static_cast<size_t>(l) * 3 * C,
             N, 3 * C, C, bf16 ? kEpiOut16 : kEpiF32, s));
    if (kv != nullptr && !decode) {  // a decode step appends in its attention kernel
      if (bf16) {
        uint16_t* kc = static_cast<uint16_t*>(kv->base) + l * kv_slab;
        launch_kv_store_16(kc, kc + kv_half, static_cast<const uint16_t*>(qkv), B, T, C, NH, kv->rows, s);
      } else {
        float* kc = static_cast<float*>(kv->base) + l * kv_slab;
        launch_kv_store_f32(kc, kc + kv_half, static_cast<const float*>(qkv), B, T, C, NH, kv->rows, s);
      }
    }
    TRY(mark(GPT2_STAGE_QKV));
    if (!decode) {
      if (precision == GPT2_FP32) {
        TRY(launch_attention_f32(static_cast<float*>(att), static_cast<const float*>(qkv), B, T, C, NH, s));
      } else if (precision == GPT2_TF32) {
        void* q16 = ws + wl.qkv16;
        to16(GPT2_BF16, q16, static_cast<const float*>(qkv), static_cast<long long>(N) * 3 * C, s);
        TRY(launch_attention_16(att, false, q16, kOpBF16, B, T, C, NH, s));
      } else {
        TRY(launch_attention_16(att, true, qkv, op, B, T, C, NH, s));
      }
    } else {
      if (bf16) {
        uint16_t* kc = static_cast<uint16_t*>(kv->base) + l * kv_slab;
        launch_decode_attention_16(att, true, qkv, kc, kc + kv_half, op, B, C, NH, decode_pos, pos_arr, kv->rows, s);
      } else {
        float* kc = static_cast<float*>(kv->base) + l * kv_slab;
        launch_decode_attention_f32(static_cast<float*>(att), static_cast<const float*>(qkv), kc, kc + kv_half, B, C,
                                    NH, decode_pos, pos_arr, kv->rows, s);
      }
    }
    TRY(check_launch());
    TRY(mark(GPT2_STAGE_ATTENTION));
    TRY(gemm(precision, bf16 ? y16 : static_cast<void*>(x), att, wmat(po.attprojw, ko.attprojw, CC, l),
             params + po.attprojb + static_cast<size_t>(l) * C, N, C, C, bf16 ? kEpiOut16 : kEpiResidF32, s));
    TRY(mark(GPT2_STAGE_ATTPROJ));
    if (bf16)
      resid_layernorm(po.ln2w + static_cast<size_t>(l) * C, po.ln2b + static_cast<size_t>(l) * C, true);
    else
      layernorm(ln, x, po.ln2w + static_cast<size_t>(l) * C, po.ln2b + static_cast<size_t>(l) * C);
    TRY(mark(GPT2_STAGE_LN2));
    TRY(gemm(precision, fch, ln, wmat(po.fcw, ko.fcw, 4 * CC, l), params + po.fcb + static_cast<size_t>(l) * 4 * C, N,
             4 * C, C, kEpiGelu16, s));
    TRY(mark(GPT2_STAGE_FC));
    TRY(gemm(precision, bf16 ? y16 : static_cast<void*>(x), fch, wmat(po.fcprojw, ko.fcprojw, 4 * CC, l),
             params + po.fcprojb + static_cast<size_t>(l) * C, N, C, 4 * C, bf16 ? kEpiOut16 : kEpiResidF32, s));
    TRY(mark(GPT2_STAGE_FCPROJ));
  }
  if (bf16 && L > 0)  // the residual stream is not read after the final LayerNorm
    resid_layernorm(po.lnfw, po.lnfb, false);
  else
    layernorm(ln, x, po.lnfw, po.lnfb);
  TRY(mark(GPT2_STAGE_LNF));
  const void* wte = bf16 ? static_cast<const void*>(pk + ko.wte) : static_cast<const void*>(params + po.wte);
  float2* stats = reinterpret_cast<float2*>(ws + wl.stats);
  if (precision == GPT2_FP32)
    TRY(gemm(precision, logits, ln, wte, nullptr, N, Vp, C, kEpiF32, s));
  else
    TRY(launch_gemm_logits(logits, stats, ln, wte, N, Vp, C, V, op, s));
  TRY(mark(GPT2_STAGE_LMHEAD));
  if (probs != nullptr) {
    if (precision == GPT2_FP32)
      launch_softmax(probs, probs_type, logits, N, V, Vp, s);
    else
      launch_softmax_from_stats(probs, probs_type, logits, stats, logits_stat_blocks(Vp), N, V, Vp, s);
  }
  TRY(check_launch());
  TRY(mark(GPT2_STAGE_SOFTMAX));
  return GPT2_OK;
}

int gpt2_forward_ex(const GPT2Config* cfg, const float* params, const void* packed, const int* tok, int B, int T,
                    float* logits, void* probs, int probs_type, void* kvcache, void* workspace, size_t ws_bytes,
                    int precision, void* stream) {
  TRY(check_config(cfg));
  RETURN_IF(!params || !tok || !logits || !workspace || !valid_precision(precision) || !valid_probs_type(probs_type),
            GPT2_ERR_ARG);
  RETURN_IF(B <= 0 || T <= 0, GPT2_ERR_ARG);
  RETURN_IF(T > cfg->max_seq_len, GPT2_ERR_SHAPE);
  TRY(check_attention_shape(cfg->channels, cfg->num_heads));
  RETURN_IF(is16(precision) && packed == nullptr, GPT2_ERR_ARG);
  RETURN_IF(!aligned16(params) || !aligned16(logits) || (probs && !aligned16(probs)) ||
                (kvcache && !aligned16(kvcache)) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                (packed && (reinterpret_cast<uintptr_t>(packed) & 255u) != 0),
            GPT2_ERR_ALIGN);
  PdlScope pdl(is16(precision));  // every kernel of the 16-bit pass waits for its predecessor itself
  const KVLayout kv = dense_kv(cfg, kvcache, B);
  return run_forward(cfg, params, packed, tok, B, T, false, 0, nullptr, logits, probs,
                     kvcache != nullptr ? &kv : nullptr, workspace, ws_bytes, precision, as_stream(stream), nullptr,
                     probs_type);
}

int gpt2_forward(const GPT2Config* cfg, const float* params, const void* packed, const int* tok, int B, int T,
                 float* logits, float* probs, void* kvcache, void* workspace, size_t ws_bytes, int precision,
                 void* stream) {
  return gpt2_forward_ex(cfg, params, packed, tok, B, T, logits, probs, GPT2_PROBS_F32, kvcache, workspace, ws_bytes,
                         precision, stream);
}

int gpt2_forward_profile(const GPT2Config* cfg, const float* params, const void* packed, const int* tok, int B, int T,
                         float* logits, void* probs, int probs_type, void* workspace, size_t ws_bytes, int precision,
                         void* stream, float* stage_ms, int n_stages) {
  TRY(check_config(cfg));
  RETURN_IF(!params || !tok || !logits || !workspace || !stage_ms || !valid_precision(precision) ||
                !valid_probs_type(probs_type),
            GPT2_ERR_ARG);
  RETURN_IF(B <= 0 || T <= 0 || n_stages <= 0, GPT2_ERR_ARG);
  RETURN_IF(T > cfg->max_seq_len, GPT2_ERR_SHAPE);
  TRY(check_attention_shape(cfg->channels, cfg->num_heads));
  RETURN_IF(is16(precision) && packed == nullptr, GPT2_ERR_ARG);
  RETURN_IF(!aligned16(params) || !aligned16(logits) || (probs && !aligned16(probs)) ||
                (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                (packed && (reinterpret_cast<uintptr_t>(packed) & 255u) != 0),
            GPT2_ERR_ALIGN);
  PdlScope pdl(is16(precision));  // the kernels gpt2_forward launches, launched the same way
  StageProfiler prof{as_stream(stream), {}, {}};
  int rc = prof.begin();
  if (rc == GPT2_OK)
    rc = run_forward(cfg, params, packed, tok, B, T, false, 0, nullptr, logits, probs, nullptr, workspace, ws_bytes,
                     precision, as_stream(stream), &prof, probs_type);
  const int rc2 = prof.finish(stage_ms, n_stages);
  return rc != GPT2_OK ? rc : rc2;
}

int gpt2_decode_step(const GPT2Config* cfg, const float* params, const void* packed, void* kvcache, const int* tok,
                     int B, int pos, float* logits, float* probs, void* workspace, size_t ws_bytes, int precision,
                     void* stream) {
  TRY(check_config(cfg));
  RETURN_IF(!params || !tok || !logits || !workspace || !kvcache || !valid_precision(precision), GPT2_ERR_ARG);
  RETURN_IF(B <= 0, GPT2_ERR_ARG);
  RETURN_IF(pos < 0 || pos >= cfg->max_seq_len, GPT2_ERR_SHAPE);
  TRY(check_attention_shape(cfg->channels, cfg->num_heads));
  RETURN_IF(is16(precision) && packed == nullptr, GPT2_ERR_ARG);
  RETURN_IF(!aligned16(params) || !aligned16(logits) || (probs && !aligned16(probs)) || !aligned16(kvcache) ||
                (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                (packed && (reinterpret_cast<uintptr_t>(packed) & 255u) != 0),
            GPT2_ERR_ALIGN);
  PdlScope pdl(is16(precision));  // every kernel of the 16-bit step waits for its predecessor itself
  const KVLayout kv = dense_kv(cfg, kvcache, B);
  return run_forward(cfg, params, packed, tok, B, 1, true, pos, nullptr, logits, probs, &kv, workspace, ws_bytes,
                     precision, as_stream(stream));
}

size_t gpt2_paged_kvcache_size(const GPT2Config* cfg, int num_blocks, int block_size, int precision) {
  if (check_config(cfg) != GPT2_OK || num_blocks <= 0 || log2_exact(block_size) < 0 || !valid_precision(precision))
    return 0;
  return static_cast<size_t>(cfg->num_layers) * paged_layer_elems(cfg, num_blocks, block_size) *
         kv_elem_bytes(precision);
}

int gpt2_prefill_paged(const GPT2Config* cfg, const float* params, const void* packed, const int* tok, int B, int T,
                       float* logits, float* probs, const GPT2PagedKVCache* kvc, void* workspace, size_t ws_bytes,
                       int precision, void* stream) {
  TRY(check_config(cfg));
  RETURN_IF(!params || !tok || !logits || !workspace || !valid_precision(precision), GPT2_ERR_ARG);
  RETURN_IF(B <= 0 || T <= 0, GPT2_ERR_ARG);
  RETURN_IF(T > cfg->max_seq_len, GPT2_ERR_SHAPE);
  TRY(check_attention_shape(cfg->channels, cfg->num_heads));
  RETURN_IF(is16(precision) && packed == nullptr, GPT2_ERR_ARG);
  KVLayout kv;
  TRY(paged_kv(cfg, kvc, T, &kv));
  RETURN_IF(!aligned16(params) || !aligned16(logits) || (probs && !aligned16(probs)) ||
                (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                (packed && (reinterpret_cast<uintptr_t>(packed) & 255u) != 0),
            GPT2_ERR_ALIGN);
  PdlScope pdl(is16(precision));
  return run_forward(cfg, params, packed, tok, B, T, false, 0, nullptr, logits, probs, &kv, workspace, ws_bytes,
                     precision, as_stream(stream));
}

int gpt2_decode_step_paged(const GPT2Config* cfg, const float* params, const void* packed,
                           const GPT2PagedKVCache* kvc, const int* tok, const int* pos, int B, float* logits,
                           float* probs, void* workspace, size_t ws_bytes, int precision, void* stream) {
  TRY(check_config(cfg));
  RETURN_IF(!params || !tok || !pos || !logits || !workspace || !valid_precision(precision), GPT2_ERR_ARG);
  RETURN_IF(B <= 0, GPT2_ERR_ARG);
  TRY(check_attention_shape(cfg->channels, cfg->num_heads));
  RETURN_IF(is16(precision) && packed == nullptr, GPT2_ERR_ARG);
  KVLayout kv;
  TRY(paged_kv(cfg, kvc, 0, &kv));
  RETURN_IF(!aligned16(params) || !aligned16(logits) || (probs && !aligned16(probs)) ||
                (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                (packed && (reinterpret_cast<uintptr_t>(packed) & 255u) != 0),
            GPT2_ERR_ALIGN);
  PdlScope pdl(is16(precision));
  return run_forward(cfg, params, packed, tok, B, 1, true, 0, pos, logits, probs, &kv, workspace, ws_bytes, precision,
                     as_stream(stream));
}

int gpt2_get_error(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) {
    g_last_cuda_error = cudaGetErrorString(cudaGetLastError());
    return GPT2_ERR_CUDA;
  }
  unsigned int w = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&w, g_error_word, sizeof(w)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) {
    g_last_cuda_error = cudaGetErrorString(cudaGetLastError());
    return GPT2_ERR_CUDA;
  }
  return static_cast<int>(w);
}

const char* gpt2_strerror(int code) {
  switch (code) {
    case GPT2_OK: return "ok";
    case GPT2_ERR_ARG: return "invalid argument";
    case GPT2_ERR_SHAPE: return "unsupported or inconsistent shape";
    case GPT2_ERR_ALIGN: return "pointer not aligned";
    case GPT2_ERR_WORKSPACE: return "workspace or buffer too small";
    case GPT2_ERR_CUDA: return "CUDA error";
    case GPT2_ERR_DEVICE: return "device-detected fault";
    case GPT2_ERR_UNSUPPORTED: return "unsupported configuration";
  }
  return "unknown error";
}

const char* gpt2_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

size_t gpt2_train_workspace_size(const GPT2Config* cfg, int B, int T, int precision) {
  if (check_config(cfg) != GPT2_OK || B <= 0 || T <= 0 || (precision != GPT2_FP32 && precision != GPT2_TF32))
    return 0;
  return train_layout(cfg, B, T).total;
}

int gpt2_forward_backward(const GPT2Config* cfg, const float* params, float* grads, const int* tok,
                          const int* targets, int B, int T, float* loss, void* workspace, size_t ws_bytes,
                          int precision, void* stream) {
  TRY(check_config(cfg));
  RETURN_IF(!params || !grads || !tok || !targets || !loss || !workspace, GPT2_ERR_ARG);
  RETURN_IF(B <= 0 || T <= 0, GPT2_ERR_ARG);
  RETURN_IF(precision != GPT2_FP32 && precision != GPT2_TF32, GPT2_ERR_UNSUPPORTED);
  RETURN_IF(T > cfg->max_seq_len, GPT2_ERR_SHAPE);
  TRY(check_attention_shape(cfg->channels, cfg->num_heads));
  // tf32 operands: every K-major row of a GEMM operand is a whole number of
  // 16-byte units (the reductions run over C, 4C, Vp and the B*T tokens)
  RETURN_IF(precision == GPT2_TF32 && (cfg->channels % 8 != 0 || (B * T) % 4 != 0), GPT2_ERR_SHAPE);
  RETURN_IF(!aligned16(params) || !aligned16(grads) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0,
            GPT2_ERR_ALIGN);
  const TrainLayout tl = train_layout(cfg, B, T);
  RETURN_IF(ws_bytes < tl.total, GPT2_ERR_WORKSPACE);
  cudaStream_t s = as_stream(stream);
  const int C = cfg->channels, L = cfg->num_layers, NH = cfg->num_heads, V = cfg->vocab_size;
  const int Vp = cfg->padded_vocab_size, maxT = cfg->max_seq_len;
  const int N = B * T;
  const size_t NC = static_cast<size_t>(N) * C, CC = static_cast<size_t>(C) * C;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto buf = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  float *xin = buf(tl.xin), *xmid = buf(tl.xmid), *ln1 = buf(tl.ln1), *ln2 = buf(tl.ln2);
  float *ln1m = buf(tl.ln1m), *ln1r = buf(tl.ln1r), *ln2m = buf(tl.ln2m), *ln2r = buf(tl.ln2r);
  float *qkv = buf(tl.qkv), *att = buf(tl.att), *fc = buf(tl.fc), *fcg = buf(tl.fcg);
  float *lnf = buf(tl.lnf), *lnfm = buf(tl.lnfm), *lnfr = buf(tl.lnfr), *logits = buf(tl.logits);
  float *losses = buf(tl.losses), *dx = buf(tl.dx), *dh = buf(tl.dh), *dt = buf(tl.dt);
  float *dt2 = buf(tl.dt2), *dqkv = buf(tl.dqkv), *tA = buf(tl.tA), *tB = buf(tl.tB), *Wt = buf(tl.Wt);
  float *part = buf(tl.part), *attn = buf(tl.attn), *lse = buf(tl.lse), *splitk = buf(tl.splitk);
  // the tf32 mode's bf16 copies of each layer's qkv, made by the forward and
  // read again by the backward, and of the attention output's gradient, in
  // the backward's scratch (free while it is used)
  auto qkv16 = [&](int l) { return static_cast<void*>(ws + tl.qkv16 + l * 3 * NC * 2); };
  void* do16 = ws + tl.dt;
  // tf32 with head size 64: attention forward and backward on tcgen05, the
  // forward keeping each row's log-sum-exp (per layer) for the backward
  const bool attn_tc = precision == GPT2_TF32 && C / NH == 64;
  const size_t SL = static_cast<size_t>(B) * NH * attn_bwd_padded_len(T);
  const ParamOffsets po = param_offsets(cfg);
  auto P = [&](size_t off) { return params + off; };
  auto G = [&](size_t off) { return grads + off; };
  // out = resid + A W^T + bias over the N rows: on tf32 tensor cores the
  // residual is added in the GEMM's epilogue (the same two fp32 additions
  // as a separate pass, without writing and reading the product); else the
  // product, then the residual add in place
  auto gemm_residual = [&](float* out, const float* resid, const float* A, const float* W, const float* bias, int OC,
                           int IC) -> int {
    if (precision == GPT2_TF32 && N > kSkinnyMaxRows)
      return launch_gemm_tc(out, A, W, bias, N, OC, IC, kEpiResidF32, kOpTF32, s, resid);
    TRY(gemm(precision, out, A, W, bias, N, OC, IC, kEpiF32, s));
    launch_residual(out, resid, out, static_cast<int>(static_cast<size_t>(N) * OC), s);
    return check_launch();
  };
  // ---------------------------------------------------------------- forward
  launch_encoder(xin, tok, P(po.wte), P(po.wpe), N, T, C, V, s);
  for (int l = 0; l < L; ++l) {
    float* x = xin + l * NC;
    launch_layernorm_f32(ln1 + l * NC, ln1m + static_cast<size_t>(l) * N, ln1r + static_cast<size_t>(l) * N, x,
                         P(po.ln1w) + l * C, P(po.ln1b) + l * C, N, C, s);
    TRY(gemm(precision, qkv + l * 3 * NC, ln1 + l * NC, P(po.qkvw) + l * 3 * CC, P(po.qkvb) + l * 3 * C, N, 3 * C, C,
             kEpiF32, s));
    if (precision == GPT2_FP32) {
      TRY(launch_attention_f32(att + l * NC, qkv + l * 3 * NC, B, T, C, NH, s));
    } else {  // as in the forward pass's tf32 mode: the bf16 tensor-core kernel on a bf16 copy of qkv
      to16(GPT2_BF16, qkv16(l), qkv + l * 3 * NC, static_cast<long long>(3 * NC), s);
      if (attn_tc)
        TRY(launch_attention_tc05(att + l * NC, false, qkv16(l), kOpBF16, B, T, C, NH, s, lse + l * SL));
      else
        TRY(launch_attention_16(att + l * NC, false, qkv16(l), kOpBF16, B, T, C, NH, s));
    }
    TRY(gemm_residual(xmid + l * NC, x, att + l * NC, P(po.attprojw) + l * CC, P(po.attprojb) + l * C, C, C));
    launch_layernorm_f32(ln2 + l * NC, ln2m + static_cast<size_t>(l) * N, ln2r + static_cast<size_t>(l) * N,
                         xmid + l * NC, P(po.ln2w) + l * C, P(po.ln2b) + l * C, N, C, s);
    if (precision == GPT2_TF32 && N > kSkinnyMaxRows) {  // pre-activation and GELU from one epilogue
      TRY(launch_gemm_tc(fc + l * 4 * NC, ln2 + l * NC, P(po.fcw) + l * 4 * CC, P(po.fcb) + l * 4 * C, N, 4 * C, C,
                         kEpiGeluDualF32, kOpTF32, s, fcg + l * 4 * NC));
    } else {
      TRY(gemm(precision, fc + l * 4 * NC, ln2 + l * NC, P(po.fcw) + l * 4 * CC, P(po.fcb) + l * 4 * C, N, 4 * C, C,
               kEpiF32, s));
      launch_gelu(fcg + l * 4 * NC, fc + l * 4 * NC, static_cast<int>(4 * NC), s);
    }
    TRY(gemm_residual(xin + (l + 1) * NC, xmid + l * NC, fcg + l * 4 * NC, P(po.fcprojw) + l * 4 * CC,
                      P(po.fcprojb) + l * C, C, 4 * C));
  }
  launch_layernorm_f32(lnf, lnfm, lnfr, xin + L * NC, P(po.lnfw), P(po.lnfb), N, C, s);
  TRY(gemm(precision, logits, lnf, P(po.wte), nullptr, N, Vp, C, kEpiF32, s));
  launch_crossentropy(logits, losses, loss, targets, N, V, Vp, s);  // logits become dL/dlogits
  TRY(check_launch());
  // --------------------------------------------------------------- backward
  // y = x W^T + b with x [N,K], W [OC,K]: dx = dy W (set), dW = dy^T x (set),
  // db = column sums of dy; the GEMM kernels take K-major operands, so W,
  // dy and x are transposed first
  // dinp = dy W (times GELU'(gelu_in) when given: the gradient through the
  // GELU that produced x, computed in the tf32 GEMM's epilogue, else by a
  // separate pass from the scratch dt), dW = dy^T x, db = column sums of dy
  auto mm_bwd = [&](float* dinp, float* dW, float* db, const float* dy, const float* x, const float* W, int OC,
                    int K, const float* gelu_in = nullptr) -> int {
    launch_transpose(Wt, W, OC, K, s);  // [K][OC]
    if (gelu_in != nullptr && precision == GPT2_TF32 && N > kSkinnyMaxRows) {
      TRY(launch_gemm_tc(dinp, dy, Wt, nullptr, N, K, OC, kEpiGeluBwdF32, kOpTF32, s, gelu_in));
    } else if (gelu_in != nullptr) {  // dy W into the scratch dt (4NC floats), then through the GELU
      TRY(gemm(precision, dt, dy, Wt, nullptr, N, K, OC, kEpiF32, s));
      launch_gelu_backward(dinp, gelu_in, dt, static_cast<long long>(N) * K, s);
    } else {
      TRY(gemm(precision, dinp, dy, Wt, nullptr, N, K, OC, kEpiF32, s));
    }
    launch_transpose(tA, dy, N, OC, s);  // [OC][N]
    launch_transpose(tB, x, N, K, s);    // [K][N]
    if (precision == GPT2_FP32) {
      TRY(gemm(precision, dW, tA, tB, nullptr, OC, K, N, kEpiF32, s));
    } else {  // an [OC][K] product over all N tokens: few, long tiles, so the K range is split
      TRY(launch_gemm_tc_splitk(dW, splitk, kSplitkFloats(C), tA, tB, OC, K, N, op_of(precision), s));
    }
    if (db != nullptr) launch_column_sum(db, part, dy, N, OC, false, s);
    return check_launch();
  };
  TRY(mm_bwd(dh, G(po.wte), nullptr, logits, lnf, P(po.wte), Vp, C));  // the tied LM head
  launch_layernorm_backward(dx, G(po.lnfw), G(po.lnfb), part, dh, xin + L * NC, P(po.lnfw), lnfm, lnfr, N, C, false,
                            s);
  for (int l = L - 1; l >= 0; --l) {
    // x_out = x_mid + fcproj(GELU(fc(LN2(x_mid)))); dx = dL/dx_out
    TRY(mm_bwd(dt2, G(po.fcprojw) + l * 4 * CC, G(po.fcprojb) + l * C, dx, fcg + l * 4 * NC,
               P(po.fcprojw) + l * 4 * CC, C, 4 * C, fc + l * 4 * NC));
    TRY(mm_bwd(dh, G(po.fcw) + l * 4 * CC, G(po.fcb) + l * 4 * C, dt2, ln2 + l * NC, P(po.fcw) + l * 4 * CC, 4 * C,
               C));
    launch_layernorm_backward(dx, G(po.ln2w) + l * C, G(po.ln2b) + l * C, part, dh, xmid + l * NC, P(po.ln2w) + l * C,
                              ln2m + static_cast<size_t>(l) * N, ln2r + static_cast<size_t>(l) * N, N, C, true, s);
    // x_mid = x_in + attproj(attention(qkv(LN1(x_in)))); dx = dL/dx_mid
    TRY(mm_bwd(dh, G(po.attprojw) + l * CC, G(po.attprojb) + l * C, dx, att + l * NC, P(po.attprojw) + l * CC, C, C));
    if (attn_tc) {
      launch_attn_bwd_prep(do16, attn, lse + l * SL, dh, att + l * NC, B, T, C, NH, s);
      TRY(launch_attention_backward_tc05(dqkv, qkv16(l), do16, lse + l * SL, attn, B, T, C, NH, s));
    } else {
      TRY(launch_attention_backward(dqkv, dh, qkv + l * 3 * NC, att + l * NC, attn,
                                    attn + static_cast<size_t>(B) * NH * T, B, T, C, NH, s));
    }
    TRY(mm_bwd(dh, G(po.qkvw) + l * 3 * CC, G(po.qkvb) + l * 3 * C, dqkv, ln1 + l * NC, P(po.qkvw) + l * 3 * CC,
               3 * C, C));
    launch_layernorm_backward(dx, G(po.ln1w) + l * C, G(po.ln1b) + l * C, part, dh, xin + l * NC, P(po.ln1w) + l * C,
                              ln1m + static_cast<size_t>(l) * N, ln1r + static_cast<size_t>(l) * N, N, C, true, s);
  }
  // the encoder: x = wte[tok] + wpe[t]; the position rows past T get none
  if (T < maxT) {
    const cudaError_t e = cudaMemsetAsync(G(po.wpe) + static_cast<size_t>(T) * C, 0,
                                          static_cast<size_t>(maxT - T) * C * sizeof(float), s);
    if (e != cudaSuccess) return note_cuda_error(e);
  }
  launch_encoder_backward(G(po.wte), G(po.wpe), dx, tok, B, T, C, V, s);
  return check_launch();
}

int gpt2_adamw(float* params, const float* grads, float* m, float* v, size_t n, float lr, float beta1, float beta2,
               float eps, float weight_decay, int t, void* stream) {
  RETURN_IF(!params || !grads || !m || !v || t < 1, GPT2_ERR_ARG);
  RETURN_IF(!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f) || !(eps > 0.f), GPT2_ERR_ARG);
  if (n == 0) return GPT2_OK;
  launch_adamw(params, grads, m, v, static_cast<long long>(n), lr, beta1, beta2, eps, weight_decay, t,
               as_stream(stream));
  return check_launch();
}

}  // extern "C"
