// C-ABI entry points of libgpt2gb (declared in include/gpt2gb.h): argument
// validation, workspace carving, and the order of kernel launches of the
// GPT-2 Pre-LN forward, block, MLP and decode step.
//
// Block dataflow ("Hidden State 如何流过 GPT-2 Block", section "GPT-2 Block";
// "逐行拆GPT-2源码", GPT2Block.forward):
//   a   = LN_1(x)                          layernorm (fused with the
//                                          embedding for the first block)
//   qkv = a W_qkv + b_qkv                  GEMM, epilogue + bias
//   o   = causal attention(qkv)            attention kernel (scores / 8, and
//                                          / (layer + 1) with that switch)
//   h   = x + o W_o + b_o                  GEMM, epilogue + bias + residual
//   a   = LN_2(h)                          layernorm
//   g   = gelu_new(a W_fc + b_fc)          GEMM, epilogue gelu_new(+ bias)
//                                          (the exact GELU with that switch)
//   x'  = h + g W_proj + b_proj            GEMM, epilogue + bias + residual
// then LN_f and the tied lm_head (GEMM against wte [V, D], no bias).
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace gpt2 {

__device__ unsigned g_error_word = 0;

namespace {

constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices] = {nullptr};
int g_sms[kMaxDevices] = {0};
std::mutex g_mu;

int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

}  // namespace

unsigned* device_error_word() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  if (!g_err_ptr[d]) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[d]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) g_err_ptr[d] = static_cast<unsigned*>(p);
    }
  }
  return g_err_ptr[d];
}

int num_sms() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 1;
  if (!g_sms[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 1;
  }
  return g_sms[d];
}

}  // namespace gpt2

using namespace gpt2;

namespace {

constexpr int kAbiVersion = 4;

// ------------------------------------------------------------- profiler
struct ProfRec {
  int name_id;
  int ev0;  // events ev0 (start) and ev0 + 1 (end)
  double flops, bytes;
};

struct Profiler {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> ev;
  int next_ev = 0;
  std::vector<ProfRec> recs;
  std::vector<std::string> names;

  void release() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    ev.clear();
    recs.clear();
    names.clear();
    next_ev = 0;
  }
  int name_id(const char* n) {
    for (size_t i = 0; i < names.size(); ++i)
      if (names[i] == n) return static_cast<int>(i);
    names.emplace_back(n);
    return static_cast<int>(names.size() - 1);
  }
};
Profiler g_prof;

// Brackets one kernel launch with events on its stream while profiling is on.
class ProfScope {
 public:
  ProfScope(const char* name, double flops, double bytes, cudaStream_t s) : s_(s) {
    if (!g_prof.on) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (!g_prof.on || g_prof.next_ev + 2 > static_cast<int>(g_prof.ev.size())) return;
    idx_ = g_prof.next_ev;
    g_prof.next_ev += 2;
    g_prof.recs.push_back({g_prof.name_id(name), idx_, flops, bytes});
    cudaEventRecord(g_prof.ev[idx_], s_);
  }
  ~ProfScope() {
    if (idx_ >= 0) cudaEventRecord(g_prof.ev[idx_ + 1], s_);
  }
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  cudaStream_t s_;
  int idx_ = -1;
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }
inline size_t esize(gpt2_dtype t) { return t == GPT2_F32 ? 4 : 2; }
inline bool valid_dtype(int t) { return t == GPT2_F32 || t == GPT2_BF16 || t == GPT2_F16; }
inline bool is16(gpt2_dtype t) { return t == GPT2_BF16 || t == GPT2_F16; }
inline cudaStream_t cs(gpt2_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

struct Carve {
  char* base;
  size_t off = 0;
  explicit Carve(void* p) : base(static_cast<char*>(p)) {}
  template <typename T>
  T* take(size_t count, size_t elem) {
    T* r = reinterpret_cast<T*>(base + off);
    off += align256(count * elem);
    return r;
  }
};

// Checks the shape fields of a dims struct; `need_model` adds n_layer,
// vocab and n_pos.
int check_dims(const gpt2_dims* d, bool need_model) {
  if (!d) return GPT2_ERR_ARG;
  if (!valid_dtype(d->dtype)) return GPT2_ERR_ARG;
  if (d->d_model <= 0 || d->n_head <= 0 || d->d_ff <= 0) return GPT2_ERR_ARG;
  if (!(d->eps > 0.f) || !std::isfinite(d->eps)) return GPT2_ERR_ARG;
  if (d->d_model % d->n_head != 0 || d->d_model / d->n_head != 64) return GPT2_ERR_UNSUPPORTED;
  if (d->d_model > 4096 || d->d_ff % 64 != 0 || d->d_ff > 65536) return GPT2_ERR_UNSUPPORTED;
  if (d->flags & ~static_cast<unsigned>(GPT2_SCALE_ATTN_BY_INVERSE_LAYER_IDX | GPT2_GELU_EXACT)) return GPT2_ERR_ARG;
  if (need_model) {
    if (d->n_layer <= 0 || d->vocab <= 0 || d->n_pos <= 0) return GPT2_ERR_ARG;
  }
  return GPT2_OK;
}

int check_block_ptrs(const gpt2_block_weights* w) {
  if (!w) return GPT2_ERR_ARG;
  const void* ps[12] = {w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_o,  w->b_o,
                        w->ln2_g, w->ln2_b, w->w_fc,  w->b_fc,  w->w_proj, w->b_proj};
  for (const void* p : ps)
    if (!p || !aligned16(p)) return GPT2_ERR_ARG;
  return GPT2_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA; }

#define GPT2_TRY(expr)                 \
  do {                                 \
    int _s = (expr);                   \
    if (_s != GPT2_OK) return _s;      \
  } while (0)
#define GPT2_CUDA(expr) GPT2_TRY(cuda_status(expr))

// ------------------------------------------------------------ launch graphs
// The multi-kernel entry points (forward, loss, training step, prefill,
// decode step) launch 60-260 kernels per call.  A call whose arguments
// (every pointer, size and the stream) equal those of an earlier call
// replays a CUDA graph captured from that earlier sequence of launches: the
// same kernels with the same parameters, launched as one graph (whose
// per-kernel launch cost on the device is lower; programmatic launch
// between the kernels is kept as graph edges).  The first call with a key
// runs eagerly (it also performs the one-time per-device set-up: kernel
// attributes, occupancy queries); the second is captured and replayed;
// later ones replay.  Calls on the legacy default stream, calls made while
// the stream is itself being captured (the caller's own graph), and calls
// while the launch profiler is on run eagerly.  A capture or instantiation
// that fails leaves that key eager.  At most kMaxGraphs keys are kept (least
// recently used evicted).
struct GraphEntry {
  std::vector<uint64_t> key;
  cudaGraphExec_t exec = nullptr;
  int state = 0;  // 1: seen once (eager), 2: graph ready, -1: eager for good
  uint64_t last_use = 0;
};
struct GraphCache {
  std::mutex mu;
  std::vector<GraphEntry> entries;
  uint64_t tick = 0;
};
GraphCache g_graphs;
constexpr size_t kMaxGraphs = 16;

struct KeyBuilder {
  std::vector<uint64_t> w;
  KeyBuilder& add(uint64_t v) {
    w.push_back(v);
    return *this;
  }
  KeyBuilder& ptr(const void* p) { return add(reinterpret_cast<uint64_t>(p)); }
  KeyBuilder& dims(const gpt2_dims* d) {
    uint32_t eps_bits;
    std::memcpy(&eps_bits, &d->eps, 4);
    return add(d->n_layer).add(d->d_model).add(d->n_head).add(d->d_ff).add(d->vocab).add(d->n_pos).add(eps_bits)
        .add(d->dtype).add(d->flags);
  }
  KeyBuilder& model(const gpt2_model_weights* m, int n_layer) {
    ptr(m->wte).ptr(m->wpe).ptr(m->lnf_g).ptr(m->lnf_b);
    for (int l = 0; l < n_layer; ++l) {
      const gpt2_block_weights& b = m->blocks[l];
      ptr(b.ln1_g).ptr(b.ln1_b).ptr(b.w_qkv).ptr(b.b_qkv).ptr(b.w_o).ptr(b.b_o);
      ptr(b.ln2_g).ptr(b.ln2_b).ptr(b.w_fc).ptr(b.b_fc).ptr(b.w_proj).ptr(b.b_proj);
    }
    return *this;
  }
};

template <typename Body>
int run_graphed(KeyBuilder& kb, cudaStream_t s, Body&& body) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (s == nullptr || s == cudaStreamLegacy || s == cudaStreamPerThread || g_prof.on ||
      cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return body(s);
  int dev = 0;
  cudaGetDevice(&dev);
  kb.add(static_cast<uint64_t>(dev)).ptr(s);
  GraphEntry* e = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_graphs.mu);
    for (GraphEntry& x : g_graphs.entries)
      if (x.key == kb.w) e = &x;
    if (e && e->state == 2) {
      e->last_use = ++g_graphs.tick;
      return cuda_status(cudaGraphLaunch(e->exec, s));
    }
    if (!e) {
      if (g_graphs.entries.size() >= kMaxGraphs) {
        auto lru = std::min_element(g_graphs.entries.begin(), g_graphs.entries.end(),
                                    [](const GraphEntry& a, const GraphEntry& b) { return a.last_use < b.last_use; });
        if (lru->exec) cudaGraphExecDestroy(lru->exec);
        g_graphs.entries.erase(lru);
      }
      GraphEntry n;
      n.key = kb.w;
      n.state = 1;
      n.last_use = ++g_graphs.tick;
      g_graphs.entries.push_back(std::move(n));
      return body(s);  // first call: eager
    }
    if (e->state != 1) return body(s);
    e->state = -1;  // until the capture below succeeds
  }
  // second call with this key: capture its launches, then replay
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  bool ok = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
  if (ok) {
    const int rc = body(s);
    ok = cudaStreamEndCapture(s, &graph) == cudaSuccess && rc == GPT2_OK && graph != nullptr;
  }
  if (ok) ok = cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
  if (graph) cudaGraphDestroy(graph);
  if (!ok) {
    if (exec) cudaGraphExecDestroy(exec);
    cudaGetLastError();  // a failed capture leaves no work behind: run the calls eagerly
    return body(s);
  }
  std::lock_guard<std::mutex> lk(g_graphs.mu);
  GraphEntry* x = nullptr;
  for (GraphEntry& y : g_graphs.entries)
    if (y.key == kb.w) x = &y;
  if (!x) {  // evicted meanwhile: replay once and drop
    const int rc = cuda_status(cudaGraphLaunch(exec, s));
    cudaGraphExecDestroy(exec);
    return rc;
  }
  if (x->exec) cudaGraphExecDestroy(x->exec);
  x->exec = exec;
  x->state = 2;
  x->last_use = ++g_graphs.tick;
  return cuda_status(cudaGraphLaunch(exec, s));
}

// One linear layer on the path of dims.dtype (no argument checks).
cudaError_t linear(gpt2_dtype dt, const void* x, const void* w, const void* bias, const float* res, void* y,
                   int64_t M, int N, int K, int64_t ldy, bool w_out_in, int epi, gpt2_dtype y_t, cudaStream_t s) {
  const double e = static_cast<double>(esize(dt));
  const double bytes = (static_cast<double>(M) * K + static_cast<double>(K) * N) * e +
                       (epi != GPT2_EPI_NONE ? N * e : 0.0) +
                       (epi == GPT2_EPI_BIAS_RESIDUAL ? 4.0 * M * N : 0.0) + static_cast<double>(M) * N * esize(y_t);
  const bool rows = M <= kMaxRowsGemm;  // the few-row kernel (gemm_rows.cu)
  ProfScope prof(dt == GPT2_BF16   ? (rows ? "gemm_rows_bf16_tcgen05" : "gemm_bf16_tcgen05")
                 : dt == GPT2_F16 ? (rows ? "gemm_rows_f16_tcgen05" : "gemm_f16_tcgen05")
                                  : "gemm_f32_simt",
                 2.0 * M * N * K, bytes, s);
  if (is16(dt)) return launch_gemm_16(dt, x, w, bias, res, y, M, N, K, ldy, w_out_in, epi, y_t, s);
  return launch_gemm_f32(static_cast<const float*>(x), static_cast<const float*>(w), static_cast<const float*>(bias),
                         res, static_cast<float*>(y), M, N, K, ldy, w_out_in, epi, s);
}

// Scores q.k / sqrt(64), and with GPT2_SCALE_ATTN_BY_INVERSE_LAYER_IDX also
// / (layer + 1) ("逐行拆GPT-2源码", GPT2Config section).
float score_scale(const gpt2_dims* d, int layer) {
  const float base = 0.125f;  // 1 / sqrt(head_dim), head_dim = 64
  return (d->flags & GPT2_SCALE_ATTN_BY_INVERSE_LAYER_IDX) ? base / static_cast<float>(layer + 1) : base;
}

// The c_fc epilogue: gelu_new, or the exact GELU with GPT2_GELU_EXACT.
int mlp_epilogue(const gpt2_dims* d) { return (d->flags & GPT2_GELU_EXACT) ? GPT2_EPI_BIAS_GELU_EXACT : GPT2_EPI_BIAS_GELU; }

cudaError_t attention(gpt2_dtype dt, const void* qkv, void* out, int B, int T, int H, float scale, cudaStream_t s) {
  // causal algorithmic work: q.k and p.v over the j <= i pairs only
  const double pairs = static_cast<double>(B) * H * T * (T + 1.0) / 2.0;
  const double D = 64.0 * H;
  ProfScope prof(dt == GPT2_BF16 ? "attn_causal_bf16_tc" : dt == GPT2_F16 ? "attn_causal_f16_tc" : "attn_causal_f32",
                 4.0 * 64.0 * pairs, static_cast<double>(B) * T * 4.0 * D * esize(dt), s);
  if (is16(dt)) return launch_attention_tc(dt, qkv, out, B, T, H, scale, s);
  return launch_attention_f32(static_cast<const float*>(qkv), static_cast<float*>(out), B, T, H, scale, s);
}

cudaError_t layernorm(const void* x, const void* g, const void* b, void* y, int64_t rows, int D, float eps,
                      gpt2_dtype x_t, gpt2_dtype y_t, cudaStream_t s) {
  ProfScope prof("layernorm", 8.0 * rows * D,
                 static_cast<double>(rows) * D * (esize(x_t) + esize(y_t)) + 2.0 * D * esize(y_t), s);
  return launch_layernorm(x, g, b, y, rows, D, eps, x_t, y_t, s);
}

struct Acts {
  float* x;
  float* h;
  void* a;
  void* qkv;
  void* o;
  void* g;
};

size_t acts_bytes(const gpt2_dims* d, int64_t M) {
  const size_t e = esize(d->dtype);
  const size_t D = d->d_model, F = d->d_ff;
  return align256(M * D * 4) * 2 + align256(M * D * e) * 2 + align256(M * 3 * D * e) + align256(M * F * e);
}

Acts carve_acts(void* ws, const gpt2_dims* d, int64_t M) {
  Carve c(ws);
  const size_t e = esize(d->dtype);
  const size_t D = d->d_model, F = d->d_ff;
  Acts a;
  a.x = c.take<float>(M * D, 4);
  a.h = c.take<float>(M * D, 4);
  a.a = c.take<char>(M * D, e);
  a.qkv = c.take<char>(M * 3 * D, e);
  a.o = c.take<char>(M * D, e);
  a.g = c.take<char>(M * F, e);
  return a;
}

// The body of block `layer` (counted from 0) from `a = LN_1(x)` already
// computed; x -> x_out.  With kv_layer (16-bit paths), the layer's K and V of
// all B T positions are also written to cache slots 0..T-1 of a
// [2, B, n_head, T_max, 64] layer.
int block_body(const gpt2_dims* d, const gpt2_block_weights* w, int layer, const float* x, float* x_out, int B, int T,
               const Acts& A, cudaStream_t s, void* kv_layer = nullptr, int T_max = 0) {
  const gpt2_dtype dt = d->dtype;
  const int64_t M = static_cast<int64_t>(B) * T;
  const int D = d->d_model, F = d->d_ff, H = d->n_head;
  GPT2_CUDA(linear(dt, A.a, w->w_qkv, w->b_qkv, nullptr, A.qkv, M, 3 * D, D, 3 * D, false, GPT2_EPI_BIAS, dt, s));
  if (kv_layer) {
    ProfScope prof("kv_from_qkv", 0.0, 2.0 * M * 2 * D * esize(dt), s);
    GPT2_CUDA(launch_kv_from_qkv(dt, A.qkv, kv_layer, B, T, H, T_max, s));
  }
  GPT2_CUDA(attention(dt, A.qkv, A.o, B, T, H, score_scale(d, layer), s));
  GPT2_CUDA(linear(dt, A.o, w->w_o, w->b_o, x, A.h, M, D, D, D, false, GPT2_EPI_BIAS_RESIDUAL, GPT2_F32, s));
  GPT2_CUDA(layernorm(A.h, w->ln2_g, w->ln2_b, A.a, M, D, d->eps, GPT2_F32, dt, s));
  GPT2_CUDA(linear(dt, A.a, w->w_fc, w->b_fc, nullptr, A.g, M, F, D, F, false, mlp_epilogue(d), dt, s));
  GPT2_CUDA(linear(dt, A.g, w->w_proj, w->b_proj, A.h, x_out, M, D, F, D, false, GPT2_EPI_BIAS_RESIDUAL, GPT2_F32, s));
  return GPT2_OK;
}

int check_model(const gpt2_dims* dims, const gpt2_model_weights* w) {
  GPT2_TRY(check_dims(dims, true));
  if (!w || !w->blocks) return GPT2_ERR_ARG;
  const void* ps[4] = {w->wte, w->wpe, w->lnf_g, w->lnf_b};
  for (const void* p : ps)
    if (!p || !aligned16(p)) return GPT2_ERR_ARG;
  for (int l = 0; l < dims->n_layer; ++l) GPT2_TRY(check_block_ptrs(&w->blocks[l]));
  return GPT2_OK;
}

// The rows of a decode step: activations, then either the lm_head's argmax
// candidates (up to kMaxRowsGemm rows) or a logits buffer for argmax_rows.
size_t decode_group_ws(const gpt2_dims* d, int nb) {
  const size_t M = static_cast<size_t>(nb);
  const size_t Vp = (static_cast<size_t>(d->vocab) + 3) & ~static_cast<size_t>(3);
  const size_t head = nb <= kMaxRowsGemm ? align256(M * rows_argmax_candidates(d->vocab) * sizeof(float2))
                                         : align256(M * Vp * 4);
  return acts_bytes(d, static_cast<int64_t>(M)) + head;
}

size_t decode_ws_bytes(const gpt2_dims* d, int B) {
  return align256(static_cast<size_t>(B) * 4) + decode_group_ws(d, B);  // valid flags, then the group
}

// Buffers and phases of a decode step over rows b0 .. b0 + nb - 1 of the
// cache's B_cache sequences.
struct DecodeGroup {
  const gpt2_dims* d;
  const gpt2_model_weights* w;
  void* kv_cache;
  int B_cache, T_max, b0, nb;
  int32_t* past_len;        // + b0
  const int32_t* tokens;    // + b0
  int32_t* next_tokens;     // + b0
  float* logits;            // + b0 rows, or null
  int64_t ld;
  int* valid;               // + b0
  Acts A;
  float2* cand;             // fused argmax (nb <= kMaxRowsGemm)
  float* lg;                // otherwise the logits for argmax_rows
  cudaStream_t s;

  void carve(char* base) {
    Carve c(base);
    const size_t M = static_cast<size_t>(nb);
    const int D = d->d_model, F = d->d_ff, V = d->vocab;
    A.x = c.take<float>(M * D, 4);
    A.h = c.take<float>(M * D, 4);
    A.a = c.take<char>(M * D, 2);
    A.qkv = c.take<char>(M * 3 * D, 2);
    A.o = c.take<char>(M * D, 2);
    A.g = c.take<char>(M * F, 2);
    cand = nullptr;
    lg = nullptr;
    if (nb <= kMaxRowsGemm)
      cand = c.take<float2>(M * rows_argmax_candidates(V), sizeof(float2));
    else
      lg = c.take<float>(M * ((static_cast<size_t>(V) + 3) & ~static_cast<size_t>(3)), 4);
  }

  cudaError_t embed() {
    const int D = d->d_model;
    ProfScope prof("decode_embed_layernorm", 8.0 * nb * D, static_cast<double>(nb) * D * 10.0, s);
    return launch_decode_embed_ln(d->dtype, tokens, past_len, w->wte, w->wpe, w->blocks[0].ln1_g,
                                  w->blocks[0].ln1_b, A.x, A.a, nb, D, d->vocab, d->n_pos, T_max, d->eps, valid, s);
  }

  cudaError_t layer(int l) {
    const gpt2_dtype dt = d->dtype;
    const int D = d->d_model, F = d->d_ff, H = d->n_head;
    const gpt2_block_weights* bw = &w->blocks[l];
    cudaError_t e;
    if (l > 0 && (e = layernorm(A.x, bw->ln1_g, bw->ln1_b, A.a, nb, D, d->eps, GPT2_F32, dt, s)) != cudaSuccess)
      return e;
    if ((e = linear(dt, A.a, bw->w_qkv, bw->b_qkv, nullptr, A.qkv, nb, 3 * D, D, 3 * D, false, GPT2_EPI_BIAS, dt,
                    s)) != cudaSuccess)
      return e;
    const size_t layer_elems = static_cast<size_t>(2) * B_cache * H * static_cast<size_t>(T_max) * 64;
    void* kv_layer = static_cast<char*>(kv_cache) + l * layer_elems * esize(dt);
    {
      // the cached lengths live on the device: the bytes of this kernel are
      // left to the caller, who knows them
      ProfScope prof("decode_attn", 0.0, 0.0, s);
      if ((e = launch_decode_attention(dt, A.qkv, kv_layer, A.o, past_len, valid, nb, b0, B_cache, H, T_max,
                                       score_scale(d, l), s)) !=
          cudaSuccess)
        return e;
    }
    if ((e = linear(dt, A.o, bw->w_o, bw->b_o, A.x, A.h, nb, D, D, D, false, GPT2_EPI_BIAS_RESIDUAL, GPT2_F32, s)) !=
        cudaSuccess)
      return e;
    if ((e = layernorm(A.h, bw->ln2_g, bw->ln2_b, A.a, nb, D, d->eps, GPT2_F32, dt, s)) != cudaSuccess) return e;
    if ((e = linear(dt, A.a, bw->w_fc, bw->b_fc, nullptr, A.g, nb, F, D, F, false, mlp_epilogue(d), dt, s)) !=
        cudaSuccess)
      return e;
    return linear(dt, A.g, bw->w_proj, bw->b_proj, A.h, A.x, nb, D, F, D, false, GPT2_EPI_BIAS_RESIDUAL, GPT2_F32, s);
  }

  cudaError_t head() {
    const gpt2_dtype dt = d->dtype;
    const int D = d->d_model, V = d->vocab;
    cudaError_t e = layernorm(A.x, w->lnf_g, w->lnf_b, A.a, nb, D, d->eps, GPT2_F32, dt, s);
    if (e != cudaSuccess) return e;
    if (cand) {
      const int n_cand = rows_argmax_candidates(V);
      {
        ProfScope prof(dt == GPT2_BF16 ? "gemm_rows_bf16_tcgen05" : "gemm_rows_f16_tcgen05", 2.0 * nb * V * D,
                       (static_cast<double>(nb) + V) * D * esize(dt) + (logits ? 4.0 * nb * V : 0.0), s);
        e = launch_gemm_rows_16(dt, A.a, w->wte, nullptr, nullptr, logits, nb, V, D, logits ? ld : V, true,
                                GPT2_EPI_NONE, GPT2_F32, s, cand);
        if (e != cudaSuccess) return e;
      }
      ProfScope prof("argmax_candidates", static_cast<double>(nb) * n_cand, static_cast<double>(nb) * n_cand * 8.0,
                     s);
      return launch_argmax_candidates(cand, n_cand, nb, valid, next_tokens, past_len, s);
    }
    const int64_t Vp = (static_cast<int64_t>(V) + 3) & ~static_cast<int64_t>(3);
    float* out = logits ? logits : lg;
    const int64_t lld = logits ? ld : Vp;
    e = linear(dt, A.a, w->wte, nullptr, nullptr, out, nb, V, D, lld, true, GPT2_EPI_NONE, GPT2_F32, s);
    if (e != cudaSuccess) return e;
    ProfScope prof("argmax_rows", static_cast<double>(nb) * V, static_cast<double>(nb) * V * 4.0, s);
    return launch_argmax_rows(out, lld, nb, V, valid, next_tokens, past_len, s);
  }
};


// Embedding, the n_layer blocks and ln_f: A.a = LN_f(x_L) (type dims.dtype).
// With kv_cache ([n_layer, 2, B, n_head, T_max, 64]) every layer's K and V
// are kept in it; with lnf = false the ln_f step is left out.
int forward_to_lnf(const gpt2_dims* dims, const gpt2_model_weights* w, const int32_t* tokens, int B, int T,
                   const Acts& A, cudaStream_t s, void* kv_cache = nullptr, int T_max = 0, bool lnf = true) {
  const int64_t M = static_cast<int64_t>(B) * T;
  const gpt2_dtype dt = dims->dtype;
  const int D = dims->d_model;
  {
    ProfScope prof("embed_layernorm", 8.0 * M * D, static_cast<double>(M) * (4.0 + D * (2.0 * esize(dt) + 4.0 + esize(dt))),
                   s);
    GPT2_CUDA(launch_embed_ln(tokens, w->wte, w->wpe, w->blocks[0].ln1_g, w->blocks[0].ln1_b, A.x, A.a, B, T, D,
                              dims->vocab, dims->eps, dt, s));
  }
  for (int l = 0; l < dims->n_layer; ++l) {
    const gpt2_block_weights* bw = &w->blocks[l];
    if (l > 0) GPT2_CUDA(layernorm(A.x, bw->ln1_g, bw->ln1_b, A.a, M, D, dims->eps, GPT2_F32, dt, s));
    void* kv_layer = nullptr;
    if (kv_cache)
      kv_layer = static_cast<char*>(kv_cache) +
                 static_cast<size_t>(l) * 2 * B * dims->n_head * static_cast<size_t>(T_max) * 64 * esize(dt);
    GPT2_TRY(block_body(dims, bw, l, A.x, A.x, B, T, A, s, kv_layer, T_max));
  }
  if (lnf) GPT2_CUDA(layernorm(A.x, w->lnf_g, w->lnf_b, A.a, M, D, dims->eps, GPT2_F32, dt, s));
  return GPT2_OK;
}

// Prefill workspace after the [B T]-row activations: valid flags, the last
// rows (fp32 and 16-bit) and the head's argmax candidates or logits.
size_t prefill_extra_bytes(const gpt2_dims* d, int B) {
  const size_t b = static_cast<size_t>(B);
  const size_t Vp = (static_cast<size_t>(d->vocab) + 3) & ~static_cast<size_t>(3);
  size_t n = align256(b * 4) + align256(b * d->d_model * 4) + align256(b * d->d_model * 2);
  n += B <= kMaxRowsGemm ? align256(b * rows_argmax_candidates(d->vocab) * sizeof(float2)) : align256(b * Vp * 4);
  return n;
}

// The loss path fuses log-sum-exp into the lm_head GEMM (16-bit, more than
// kMaxRowsGemm rows); otherwise it writes fp32 logits into the workspace and
// reduces them.
bool loss_fused(const gpt2_dims* d, int64_t M) { return is16(d->dtype) && M > kMaxRowsGemm; }
int64_t loss_ld(const gpt2_dims* d) { return (static_cast<int64_t>(d->vocab) + 3) / 4 * 4; }
size_t loss_extra_bytes(const gpt2_dims* d, int64_t M) {
  const size_t m = static_cast<size_t>(M);
  size_t b = align256(m * 4) * 2;  // target logits, per-position loss scratch
  if (loss_fused(d, M))
    b += align256(m * lse_max_partials(d->vocab) * sizeof(float2));
  else
    b += align256(m * sizeof(float2)) + align256(m * loss_ld(d) * 4);
  return b;
}

// ------------------------------------------------------- block backward
// Workspace of gpt2_block_backward (fp32): the recomputed forward
// intermediates, the gradients between the steps, the LayerNorm products
// and the attention row statistics.
struct BwdActs {
  float *a, *qkv, *o, *h, *a2, *u, *g;        // forward: LN_1(x), c_attn, attention, h, LN_2(h), c_fc, act
  float *dg, *du, *da2, *dh, *dout, *dqkv, *da;  // backward
  float *prod, *lse, *delta;
  float* colpart;  // column-sum partials
};

size_t bwd_ws_bytes(const gpt2_dims* d, int B, int T) {
  const size_t M = static_cast<size_t>(B) * T, D = d->d_model, F = d->d_ff, H = d->n_head;
  const size_t rows_d = align256(M * D * 4), rows_3d = align256(M * 3 * D * 4), rows_f = align256(M * F * 4);
  const size_t stats = align256(static_cast<size_t>(B) * H * T * 4);
  return rows_d * 9 + rows_3d * 2 + rows_f * 4 + stats * 2 +
         align256(colsum_partial_bytes(static_cast<long long>(M), static_cast<int>(std::max(3 * D, F))));
}

BwdActs carve_bwd(void* ws, const gpt2_dims* d, int B, int T) {
  Carve c(ws);
  const size_t M = static_cast<size_t>(B) * T, D = d->d_model, F = d->d_ff, H = d->n_head;
  BwdActs A;
  A.a = c.take<float>(M * D, 4);
  A.qkv = c.take<float>(M * 3 * D, 4);
  A.o = c.take<float>(M * D, 4);
  A.h = c.take<float>(M * D, 4);
  A.a2 = c.take<float>(M * D, 4);
  A.u = c.take<float>(M * F, 4);
  A.g = c.take<float>(M * F, 4);
  A.dg = c.take<float>(M * F, 4);
  A.du = c.take<float>(M * F, 4);
  A.da2 = c.take<float>(M * D, 4);
  A.dh = c.take<float>(M * D, 4);
  A.dout = c.take<float>(M * D, 4);
  A.dqkv = c.take<float>(M * 3 * D, 4);
  A.da = c.take<float>(M * D, 4);
  A.prod = c.take<float>(M * D, 4);
  A.lse = c.take<float>(static_cast<size_t>(B) * H * T, 4);
  A.delta = c.take<float>(static_cast<size_t>(B) * H * T, 4);
  A.colpart = c.take<float>(colsum_partial_bytes(static_cast<long long>(M), static_cast<int>(std::max(3 * D, F))) / 4,
                            4);
  return A;
}

// Recomputes the block's forward, then runs its steps backwards:
//   x' = h + c_proj2(g):  dg = dx' W_proj^T, dW_proj = g^T dx', db_proj
//   g = act(u):           du = dg act'(u)
//   u = c_fc(LN_2(h)):    da2 = du W_fc^T, dW_fc = a2^T du, db_fc
//   LN_2, residual:       dh = dx' + LN_2'(h)^T da2, dln2_g, dln2_b
//   h = x + c_proj(o):    do = dh W_o^T, dW_o = o^T dh, db_o
//   o = attention(qkv):   dqkv
//   qkv = c_attn(LN_1(x)): da = dqkv W_qkv^T, dW_qkv = a^T dqkv, db_qkv
//   LN_1, residual:       dx = dh + LN_1'(x)^T da, dln1_g, dln1_b
int block_backward_f32(const gpt2_dims* d, const gpt2_block_weights* w, int layer, const float* x, const float* dy,
                       float* dx, const gpt2_block_grads* gr, int B, int T, void* ws, cudaStream_t s) {
  const int64_t M = static_cast<int64_t>(B) * T;
  const int D = d->d_model, F = d->d_ff, H = d->n_head;
  const float eps = d->eps, sc = score_scale(d, layer);
  const bool exact = (d->flags & GPT2_GELU_EXACT) != 0;
  BwdActs A = carve_bwd(ws, d, B, T);
  auto f = [](const void* p) { return static_cast<const float*>(p); };
  // forward
  GPT2_CUDA(layernorm(x, w->ln1_g, w->ln1_b, A.a, M, D, eps, GPT2_F32, GPT2_F32, s));
  GPT2_CUDA(linear(GPT2_F32, A.a, w->w_qkv, w->b_qkv, nullptr, A.qkv, M, 3 * D, D, 3 * D, false, GPT2_EPI_BIAS,
                   GPT2_F32, s));
  GPT2_CUDA(attention(GPT2_F32, A.qkv, A.o, B, T, H, sc, s));
  GPT2_CUDA(linear(GPT2_F32, A.o, w->w_o, w->b_o, x, A.h, M, D, D, D, false, GPT2_EPI_BIAS_RESIDUAL, GPT2_F32, s));
  GPT2_CUDA(layernorm(A.h, w->ln2_g, w->ln2_b, A.a2, M, D, eps, GPT2_F32, GPT2_F32, s));
  GPT2_CUDA(linear(GPT2_F32, A.a2, w->w_fc, w->b_fc, nullptr, A.u, M, F, D, F, false, GPT2_EPI_BIAS, GPT2_F32, s));
  GPT2_CUDA(launch_gelu_f32(A.u, A.g, M * F, exact, s));
  // MLP
  GPT2_CUDA(linear(GPT2_F32, dy, w->w_proj, nullptr, nullptr, A.dg, M, F, D, F, true, GPT2_EPI_NONE, GPT2_F32, s));
  GPT2_CUDA(launch_gemm_at_f32(A.g, dy, gr->w_proj, M, F, D, s));
  GPT2_CUDA(launch_colsum(dy, false, M, D, D, A.colpart, gr->b_proj, s));
  GPT2_CUDA(launch_gelu_backward_f32(A.dg, A.u, A.du, M * F, exact, s));
  GPT2_CUDA(linear(GPT2_F32, A.du, w->w_fc, nullptr, nullptr, A.da2, M, D, F, D, true, GPT2_EPI_NONE, GPT2_F32, s));
  GPT2_CUDA(launch_gemm_at_f32(A.a2, A.du, gr->w_fc, M, D, F, s));
  GPT2_CUDA(launch_colsum(A.du, false, M, F, F, A.colpart, gr->b_fc, s));
  // LN_2 and the residual path
  GPT2_CUDA(launch_ln_backward_f32(A.da2, A.h, f(w->ln2_g), dy, A.dh, A.prod, M, D, eps, s));
  GPT2_CUDA(launch_colsum(A.prod, false, M, D, D, A.colpart, gr->ln2_g, s));
  GPT2_CUDA(launch_colsum(A.da2, false, M, D, D, A.colpart, gr->ln2_b, s));
  // attention sublayer
  GPT2_CUDA(linear(GPT2_F32, A.dh, w->w_o, nullptr, nullptr, A.dout, M, D, D, D, true, GPT2_EPI_NONE, GPT2_F32, s));
  GPT2_CUDA(launch_gemm_at_f32(A.o, A.dh, gr->w_o, M, D, D, s));
  GPT2_CUDA(launch_colsum(A.dh, false, M, D, D, A.colpart, gr->b_o, s));
  GPT2_CUDA(launch_attention_backward_f32(A.qkv, A.dout, A.dqkv, A.lse, A.delta, B, T, H, sc, s));
  GPT2_CUDA(linear(GPT2_F32, A.dqkv, w->w_qkv, nullptr, nullptr, A.da, M, D, 3 * D, D, true, GPT2_EPI_NONE,
                   GPT2_F32, s));
  GPT2_CUDA(launch_gemm_at_f32(A.a, A.dqkv, gr->w_qkv, M, D, 3 * D, s));
  GPT2_CUDA(launch_colsum(A.dqkv, false, M, 3 * D, 3 * D, A.colpart, gr->b_qkv, s));
  // LN_1 and the residual path
  GPT2_CUDA(launch_ln_backward_f32(A.da, x, f(w->ln1_g), A.dh, dx, A.prod, M, D, eps, s));
  GPT2_CUDA(launch_colsum(A.prod, false, M, D, D, A.colpart, gr->ln1_g, s));
  GPT2_CUDA(launch_colsum(A.da, false, M, D, D, A.colpart, gr->ln1_b, s));
  return GPT2_OK;
}

// ------------------------------------------------------- training step
// Buffers of gpt2_forward_backward (bf16 path).  Per layer the forward keeps
// what the backward reads (llm.c notes 5.2: the intermediates are kept):
// the block input x (fp32), LN_1 output a, qkv, the attention output o and
// its row log-sum-exp, h (fp32), LN_2 output a2, the c_fc output u and its
// GELU g.  Then x_L, LN_f(x_L), the loss buffers, and the backward scratch.
struct TrainLayer {
  float *x, *h, *lse;
  void *a, *qkv, *o, *a2, *u, *g;
};
struct TrainBufs {
  std::vector<TrainLayer> L;
  float* xL;
  void* xf;
  float *tgt, *tl, *row_lse, *logits32;
  float2* part;
  int64_t ldz;
  void* dz;
  float *dx, *dh, *dyf, *delta, *colpart, *splitk;
  size_t splitk_bytes;
  void *dxb, *dhb, *dgb, *dub, *dob, *dqkvb;
  size_t bytes;
};

// Carves the buffers from `ws` (or, with ws == nullptr, only counts bytes).
TrainBufs carve_train(void* ws, const gpt2_dims* d, int B, int T) {
  const size_t M = static_cast<size_t>(B) * T, D = d->d_model, F = d->d_ff, H = d->n_head, V = d->vocab;
  size_t off = 0;
  char* base = static_cast<char*>(ws);
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? static_cast<void*>(base + off) : nullptr;
    off += align256(bytes);
    return p;
  };
  TrainBufs t;
  t.L.resize(d->n_layer);
  for (int l = 0; l < d->n_layer; ++l) {
    TrainLayer& y = t.L[l];
    y.x = static_cast<float*>(take(M * D * 4));
    y.h = static_cast<float*>(take(M * D * 4));
    y.lse = static_cast<float*>(take(static_cast<size_t>(B) * H * T * 4));
    y.a = take(M * D * 2);
    y.qkv = take(M * 3 * D * 2);
    y.o = take(M * D * 2);
    y.a2 = take(M * D * 2);
    y.u = take(M * F * 2);
    y.g = take(M * F * 2);
  }
  t.xL = static_cast<float*>(take(M * D * 4));
  t.xf = take(M * D * 2);
  t.tgt = static_cast<float*>(take(M * 4));
  t.tl = static_cast<float*>(take(M * 4));
  t.row_lse = static_cast<float*>(take(M * 4));
  const bool fused = static_cast<int64_t>(M) > kMaxRowsGemm;
  t.part = static_cast<float2*>(take((fused ? M * lse_max_partials(d->vocab) : M) * sizeof(float2)));
  t.logits32 = fused ? nullptr : static_cast<float*>(take(M * ((V + 3) / 4 * 4) * 4));
  t.ldz = (static_cast<int64_t>(V) + 7) / 8 * 8;
  t.dz = take(M * t.ldz * 2);
  t.dx = static_cast<float*>(take(M * D * 4));
  t.dh = static_cast<float*>(take(M * D * 4));
  t.dyf = static_cast<float*>(take(M * D * 4));
  t.delta = static_cast<float*>(take(static_cast<size_t>(B) * H * T * 4));
  const size_t widest = std::max<size_t>({3 * D, F, D});
  // column-sum partials: the generic sums (bias of qkv) and those of the
  // LayerNorm and GELU backward kernels
  const long long Ml = static_cast<long long>(M);
  t.colpart = static_cast<float*>(take(std::max(colsum_partial_bytes(Ml, static_cast<int>(widest)),
                                                ln_bwd_scratch_bytes(Ml, static_cast<int>(D)))));
  {
    // fp32 partial slabs of the split-K weight-gradient products
    const int Mi = static_cast<int>(M), Di = static_cast<int>(D), Fi = static_cast<int>(F);
    size_t sk = 0;
    const int shapes[5][2] = {{Di, 3 * Di}, {Di, Di}, {Di, Fi}, {Fi, Di}, {static_cast<int>(V), Di}};
    for (const auto& sh : shapes) sk = std::max(sk, gemm_grad_scratch_bytes(sh[0], sh[1], Mi));
    t.splitk_bytes = sk;
    t.splitk = static_cast<float*>(take(sk));
  }
  t.dxb = take(M * D * 2);
  t.dhb = take(M * D * 2);
  t.dgb = take(M * F * 2);
  t.dub = take(M * F * 2);
  t.dob = take(M * D * 2);
  t.dqkvb = take(M * 3 * D * 2);
  t.bytes = off;
  return t;
}

int check_grads(const gpt2_dims* d, const gpt2_model_grads* g) {
  if (!g || !g->blocks) return GPT2_ERR_ARG;
  const void* ps[4] = {g->wte, g->wpe, g->lnf_g, g->lnf_b};
  for (const void* p : ps)
    if (!p || !aligned16(p)) return GPT2_ERR_ARG;
  for (int l = 0; l < d->n_layer; ++l) {
    const gpt2_block_grads& b = g->blocks[l];
    const float* bp[12] = {b.ln1_g, b.ln1_b, b.w_qkv, b.b_qkv, b.w_o, b.b_o,
                           b.ln2_g, b.ln2_b, b.w_fc, b.b_fc, b.w_proj, b.b_proj};
    for (const float* p : bp)
      if (!p || !aligned16(p)) return GPT2_ERR_ARG;
  }
  return GPT2_OK;
}

// One tensor-core GEMM of the backward, profiled like the forward's.
cudaError_t grad_gemm(const void* a, long long lda, bool a_mn, const void* w, long long ldw, bool w_kn, void* y,
                      long long ldy, gpt2_dtype y_t, int64_t M, int N, int K, cudaStream_t s,
                      float* scratch = nullptr, size_t scratch_bytes = 0) {
  ProfScope prof("gemm_grad_bf16_tcgen05", 2.0 * M * N * K,
                 (static_cast<double>(M) * K + static_cast<double>(K) * N) * 2.0 + static_cast<double>(M) * N * esize(y_t),
                 s);
  return launch_gemm_grad(a, lda, a_mn, w, ldw, w_kn, y, ldy, y_t, static_cast<int>(M), N, K, s, scratch,
                          scratch_bytes);
}

cudaError_t colsum(const void* in, bool in16, int64_t M, int N, float* partial, float* out, cudaStream_t s) {
  ProfScope prof("colsum", static_cast<double>(M) * N, static_cast<double>(M) * N * (in16 ? 2.0 : 4.0), s);
  return launch_colsum(in, in16, M, N, N, partial, out, s);
}

// LayerNorm backward with the column sums of dy * xhat (dgamma), dy (dbeta)
// and, when dbias is given, of dx (the bias gradient of the residual branch
// whose output is the LayerNorm's input).
cudaError_t ln_bwd(const float* dy, const float* x, const void* gamma, const float* dres, float* dx, void* dx16,
                   float* dgamma, float* dbeta, float* dbias, float* scratch, int64_t M, int D, float eps,
                   cudaStream_t s) {
  ProfScope prof("layernorm_bwd", 15.0 * M * D, static_cast<double>(M) * D * (4.0 * 3 + (dres ? 4.0 : 0.0) + 2.0), s);
  return launch_ln_bwd_sums_16(dy, x, gamma, dres, dx, dx16, dgamma, dbeta, dbias, M, D, eps, scratch, s);
}

// Forward with saved intermediates, then the mean shifted cross-entropy and
// the gradient of every parameter (the order of the backward is the reverse
// of the forward: llm.c notes 5.2-5.3; the tied lm_head and the embedding
// both add to wte: "逐行拆GPT-2源码", GPT2LMHeadModel).
int forward_backward(const gpt2_dims* d, const gpt2_model_weights* w, const int32_t* tokens, const int32_t* labels,
                     const gpt2_model_grads* gr, float* mean_loss, int B, int T, TrainBufs& t, cudaStream_t s) {
  const gpt2_dtype dt = d->dtype;
  const int64_t M = static_cast<int64_t>(B) * T;
  const int D = d->d_model, F = d->d_ff, H = d->n_head, V = d->vocab, L = d->n_layer;
  const float eps = d->eps;
  const bool exact = (d->flags & GPT2_GELU_EXACT) != 0;
  // ---- forward
  {
    ProfScope prof("embed_layernorm", 8.0 * M * D, static_cast<double>(M) * D * 10.0, s);
    GPT2_CUDA(launch_embed_ln(tokens, w->wte, w->wpe, w->blocks[0].ln1_g, w->blocks[0].ln1_b, t.L[0].x, t.L[0].a, B,
                              T, D, V, eps, dt, s));
  }
  for (int l = 0; l < L; ++l) {
    const gpt2_block_weights* bw = &w->blocks[l];
    TrainLayer& y = t.L[l];
    if (l > 0) GPT2_CUDA(layernorm(y.x, bw->ln1_g, bw->ln1_b, y.a, M, D, eps, GPT2_F32, dt, s));
    GPT2_CUDA(linear(dt, y.a, bw->w_qkv, bw->b_qkv, nullptr, y.qkv, M, 3 * D, D, 3 * D, false, GPT2_EPI_BIAS, dt, s));
    {
      const double pairs = static_cast<double>(B) * H * T * (T + 1.0) / 2.0;
      ProfScope prof("attn_causal_bf16_tc", 4.0 * 64.0 * pairs, static_cast<double>(M) * 4.0 * D * 2.0, s);
      GPT2_CUDA(launch_attention_tc(dt, y.qkv, y.o, B, T, H, score_scale(d, l), s, y.lse));
    }
    GPT2_CUDA(linear(dt, y.o, bw->w_o, bw->b_o, y.x, y.h, M, D, D, D, false, GPT2_EPI_BIAS_RESIDUAL, GPT2_F32, s));
    GPT2_CUDA(layernorm(y.h, bw->ln2_g, bw->ln2_b, y.a2, M, D, eps, GPT2_F32, dt, s));
    GPT2_CUDA(linear(dt, y.a2, bw->w_fc, bw->b_fc, nullptr, y.u, M, F, D, F, false, GPT2_EPI_BIAS, dt, s));
    {
      ProfScope prof("gelu", 8.0 * M * F, 4.0 * M * F, s);
      GPT2_CUDA(launch_gelu_fwd_16(y.u, y.g, M * F, exact, s));
    }
    float* x_next = l + 1 < L ? t.L[l + 1].x : t.xL;
    GPT2_CUDA(linear(dt, y.g, bw->w_proj, bw->b_proj, y.h, x_next, M, D, F, D, false, GPT2_EPI_BIAS_RESIDUAL, GPT2_F32,
                     s));
  }
  GPT2_CUDA(layernorm(t.xL, w->lnf_g, w->lnf_b, t.xf, M, D, eps, GPT2_F32, dt, s));
  // ---- loss: each row's log-sum-exp (kept for dz) and the mean
  int n_part = 1;
  if (t.logits32 == nullptr) {
    ProfScope prof("gemm_lse_bf16_tcgen05", 2.0 * M * V * D, (static_cast<double>(M) + V) * D * 2.0, s);
    GPT2_CUDA(launch_gemm_lse_16(dt, t.xf, w->wte, M, V, D, labels, T, t.part, t.tgt, &n_part, s));
  } else {
    const int64_t lv = (static_cast<int64_t>(V) + 3) / 4 * 4;
    GPT2_CUDA(linear(dt, t.xf, w->wte, nullptr, nullptr, t.logits32, M, V, D, lv, true, GPT2_EPI_NONE, GPT2_F32, s));
    GPT2_CUDA(launch_lse_from_logits(t.logits32, lv, M, V, labels, T, t.part, t.tgt, s));
  }
  {
    ProfScope prof("loss_reduce", 4.0 * M * n_part, 8.0 * M * n_part + 12.0 * M, s);
    GPT2_CUDA(launch_loss_rows(t.part, n_part, t.tgt, labels, B, T, V, t.row_lse, t.tl, mean_loss, s));
  }
  // ---- lm_head and LN_f
  const float inv_n = 1.f / static_cast<float>(static_cast<double>(B) * (T - 1));
  {
    ProfScope prof("gemm_dlogits_bf16_tcgen05", 2.0 * M * V * D, static_cast<double>(M) * V * 2.0, s);
    GPT2_CUDA(launch_gemm_dlogits(t.xf, w->wte, static_cast<int>(M), V, D, t.row_lse, labels, T, inv_n, t.dz, t.ldz,
                                  s));
  }
  GPT2_CUDA(grad_gemm(t.dz, t.ldz, true, t.xf, D, true, gr->wte, D, GPT2_F32, V, D, static_cast<int>(M), s, t.splitk, t.splitk_bytes));
  GPT2_CUDA(grad_gemm(t.dz, t.ldz, false, w->wte, D, true, t.dyf, D, GPT2_F32, M, D, V, s));
  // (the sums of dx: the bias gradient of the last block's MLP c_proj)
  GPT2_CUDA(ln_bwd(t.dyf, t.xL, w->lnf_g, nullptr, t.dx, t.dxb, gr->lnf_g, gr->lnf_b, gr->blocks[L - 1].b_proj,
                   t.colpart, M, D, eps, s));
  // ---- blocks, last first
  const int Mi = static_cast<int>(M);
  for (int l = L - 1; l >= 0; --l) {
    const gpt2_block_weights* bw = &w->blocks[l];
    const gpt2_block_grads* bg = &gr->blocks[l];
    TrainLayer& y = t.L[l];
    // x' = h + g W_proj + b_proj
    GPT2_CUDA(grad_gemm(t.dxb, D, false, bw->w_proj, D, false, t.dgb, F, dt, M, F, D, s));
    GPT2_CUDA(grad_gemm(y.g, F, true, t.dxb, D, true, bg->w_proj, D, GPT2_F32, F, D, Mi, s, t.splitk, t.splitk_bytes));
    {
      ProfScope prof("gelu_bwd", 21.0 * M * F, 6.0 * M * F, s);
      GPT2_CUDA(launch_gelu_bwd_sums_16(t.dgb, y.u, t.dub, M, F, exact, bg->b_fc, t.colpart, s));
    }
    // u = a2 W_fc + b_fc
    GPT2_CUDA(grad_gemm(t.dub, F, false, bw->w_fc, F, false, t.dyf, D, GPT2_F32, M, D, F, s));
    GPT2_CUDA(grad_gemm(y.a2, D, true, t.dub, F, true, bg->w_fc, F, GPT2_F32, D, F, Mi, s, t.splitk, t.splitk_bytes));
    // a2 = LN_2(h), and the residual path: dh = dx' + LN_2'(h)^T da2
    GPT2_CUDA(ln_bwd(t.dyf, y.h, bw->ln2_g, t.dx, t.dh, t.dhb, bg->ln2_g, bg->ln2_b, bg->b_o, t.colpart, M, D, eps,
                     s));
    // h = x + o W_o + b_o
    GPT2_CUDA(grad_gemm(t.dhb, D, false, bw->w_o, D, false, t.dob, D, dt, M, D, D, s));
    GPT2_CUDA(grad_gemm(y.o, D, true, t.dhb, D, true, bg->w_o, D, GPT2_F32, D, D, Mi, s, t.splitk, t.splitk_bytes));
    // o = attention(qkv)
    {
      const double pairs = static_cast<double>(B) * H * T * (T + 1.0) / 2.0;
      ProfScope prof("attn_causal_bwd_bf16_tc", 10.0 * 64.0 * pairs, static_cast<double>(M) * D * 2.0 * 8.0, s);
      GPT2_CUDA(launch_attention_backward_tc(dt, y.qkv, y.o, y.lse, t.dob, t.dqkvb, t.delta, B, T, H,
                                             score_scale(d, l), s));
    }
    // qkv = a W_qkv + b_qkv
    GPT2_CUDA(grad_gemm(t.dqkvb, 3 * D, false, bw->w_qkv, 3 * D, false, t.dyf, D, GPT2_F32, M, D, 3 * D, s));
    GPT2_CUDA(grad_gemm(y.a, D, true, t.dqkvb, 3 * D, true, bg->w_qkv, 3 * D, GPT2_F32, D, 3 * D, Mi, s, t.splitk, t.splitk_bytes));
    GPT2_CUDA(colsum(t.dqkvb, true, M, 3 * D, t.colpart, bg->b_qkv, s));
    // a = LN_1(x), and the residual path: dx = dh + LN_1'(x)^T da
    // (the sums of dx: the bias gradient of the previous block's MLP c_proj)
    GPT2_CUDA(ln_bwd(t.dyf, y.x, bw->ln1_g, t.dh, t.dx, t.dxb, bg->ln1_g, bg->ln1_b,
                     l > 0 ? gr->blocks[l - 1].b_proj : nullptr, t.colpart, M, D, eps, s));
  }
  // ---- the embedding: wte rows of the tokens used, wpe rows of the positions
  {
    ProfScope prof("embed_bwd", static_cast<double>(M) * D, static_cast<double>(M) * D * 8.0, s);
    GPT2_CUDA(launch_embed_bwd(tokens, t.dx, gr->wte, gr->wpe, B, T, D, V, d->n_pos, s));
  }
  return GPT2_OK;
}

}  // namespace

namespace gpt2 {

cudaError_t launch_mlp(gpt2_dtype dt, const void* x, const void* w_fc, const void* b_fc, const void* w_proj,
                       const void* b_proj, const float* residual, float* out, int64_t M, int D, int F, void* hidden,
                       cudaStream_t s) {
  cudaError_t e = linear(dt, x, w_fc, b_fc, nullptr, hidden, M, F, D, F, false, GPT2_EPI_BIAS_GELU, dt, s);
  if (e != cudaSuccess) return e;
  return linear(dt, hidden, w_proj, b_proj, residual, out, M, D, F, D, false,
                residual ? GPT2_EPI_BIAS_RESIDUAL : GPT2_EPI_BIAS, GPT2_F32, s);
}

// Failure-detection self-test: one thread waits, through the bounded wait
// every kernel of the library uses, on an mbarrier that nothing arrives on.
// When `limit_ns` has passed it records GPT2_ERR_TIMEOUT at its own site and
// returns, as a kernel whose producer never delivered would.
__global__ void selftest_wait_kernel(unsigned long long limit_ns, unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  if (!mbar_wait_for(b, 0, limit_ns)) record_error(err, kErrTimeout, kSiteSelfTestWait);
}

}  // namespace gpt2

extern "C" {

int gpt2_abi_version(void) { return kAbiVersion; }

const char* gpt2_status_string(int status) {
  switch (status) {
    case GPT2_OK: return "ok";
    case GPT2_ERR_ARG: return "invalid argument";
    case GPT2_ERR_UNSUPPORTED: return "unsupported shape or type";
    case GPT2_ERR_WORKSPACE: return "workspace too small";
    case GPT2_ERR_CUDA: return "CUDA error";
    case GPT2_ERR_TIMEOUT: return "device wait timed out";
    case GPT2_ERR_RANGE: return "token id or position out of range";
    default: return "unknown status";
  }
}

int gpt2_last_error(int* site) {
  if (site) *site = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return GPT2_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return GPT2_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return GPT2_ERR_CUDA;
  }
  if (site) *site = static_cast<int>(v >> 8);
  return static_cast<int>(v & 0xFFu);
}

int gpt2_selftest_wait_timeout(uint64_t limit_ns, gpt2_stream_t stream) {
  if (limit_ns == 0 || limit_ns > kWaitLimitNs) return GPT2_ERR_ARG;
  selftest_wait_kernel<<<1, 1, 0, cs(stream)>>>(static_cast<unsigned long long>(limit_ns), device_error_word());
  return cuda_status(cudaGetLastError());
}

int gpt2_layernorm(const void* x, const void* gamma, const void* beta, void* y, int64_t rows, int D, float eps,
                   gpt2_dtype x_t, gpt2_dtype y_t, gpt2_stream_t stream) {
  if (!valid_dtype(x_t) || !valid_dtype(y_t)) return GPT2_ERR_ARG;
  if (rows < 0 || D <= 0 || !(eps > 0.f) || !std::isfinite(eps)) return GPT2_ERR_ARG;
  if (D % 4 != 0 || D > 4096) return GPT2_ERR_UNSUPPORTED;
  if (rows == 0) return GPT2_OK;
  if (!x || !gamma || !beta || !y) return GPT2_ERR_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(gamma) || !aligned16(beta)) return GPT2_ERR_ARG;
  return cuda_status(layernorm(x, gamma, beta, y, rows, D, eps, x_t, y_t, cs(stream)));
}

int gpt2_linear(const void* x, const void* w, const void* bias, const float* residual, void* y, int64_t M, int N,
                int K, int64_t ldy, gpt2_weight_layout w_layout, gpt2_epilogue epilogue, gpt2_dtype dtype,
                gpt2_dtype y_t, gpt2_stream_t stream) {
  if (!valid_dtype(dtype) || !valid_dtype(y_t)) return GPT2_ERR_ARG;
  if (w_layout != GPT2_W_IN_OUT && w_layout != GPT2_W_OUT_IN) return GPT2_ERR_ARG;
  if (epilogue < GPT2_EPI_NONE || epilogue > GPT2_EPI_BIAS_GELU_EXACT) return GPT2_ERR_ARG;
  if (M < 0 || M > INT_MAX || N <= 0 || K <= 0 || ldy < N) return GPT2_ERR_ARG;
  if (K % 64 != 0) return GPT2_ERR_UNSUPPORTED;
  if (epilogue == GPT2_EPI_BIAS_RESIDUAL && y_t != GPT2_F32) return GPT2_ERR_UNSUPPORTED;
  if (dtype == GPT2_F32 && y_t != GPT2_F32) return GPT2_ERR_UNSUPPORTED;
  if (is16(dtype) && y_t != dtype && y_t != GPT2_F32) return GPT2_ERR_UNSUPPORTED;
  if (is16(dtype) && w_layout == GPT2_W_IN_OUT && N % 8 != 0) return GPT2_ERR_UNSUPPORTED;
  // the tensor-core epilogue stores 16-byte pieces: 16-byte aligned rows
  if (is16(dtype) && (ldy * static_cast<int64_t>(esize(y_t))) % 16 != 0) return GPT2_ERR_UNSUPPORTED;
  if (epilogue == GPT2_EPI_BIAS_RESIDUAL && N % 4 != 0) return GPT2_ERR_UNSUPPORTED;
  if (M == 0) return GPT2_OK;
  if (!x || !w || !y || !aligned16(x) || !aligned16(w) || !aligned16(y)) return GPT2_ERR_ARG;
  if (epilogue != GPT2_EPI_NONE && (!bias || !aligned16(bias))) return GPT2_ERR_ARG;
  if (epilogue == GPT2_EPI_BIAS_RESIDUAL && (!residual || !aligned16(residual))) return GPT2_ERR_ARG;
  return cuda_status(linear(dtype, x, w, bias, residual, y, M, N, K, ldy, w_layout == GPT2_W_OUT_IN, epilogue, y_t,
                            cs(stream)));
}

int gpt2_attention_causal(const void* qkv, void* out, int B, int T, int n_head, int head_dim, gpt2_dtype dtype,
                          gpt2_stream_t stream) {
  return gpt2_attention_causal_scaled(qkv, out, B, T, n_head, head_dim, 0.125f, dtype, stream);
}

int gpt2_attention_causal_scaled(const void* qkv, void* out, int B, int T, int n_head, int head_dim,
                                 float score_scale, gpt2_dtype dtype, gpt2_stream_t stream) {
  if (!valid_dtype(dtype) || B < 0 || T < 0 || n_head <= 0 || head_dim <= 0) return GPT2_ERR_ARG;
  if (!(score_scale > 0.f) || !std::isfinite(score_scale)) return GPT2_ERR_ARG;
  if (head_dim != 64) return GPT2_ERR_UNSUPPORTED;
  if (dtype == GPT2_F32 && T > 8192) return GPT2_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * n_head > INT_MAX || T > 65535 * 64) return GPT2_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return GPT2_OK;
  if (!qkv || !out || !aligned16(qkv) || !aligned16(out)) return GPT2_ERR_ARG;
  return cuda_status(attention(dtype, qkv, out, B, T, n_head, score_scale, cs(stream)));
}

int gpt2_attention_causal_lse(const void* qkv, void* out, float* lse, int B, int T, int n_head, int head_dim,
                              float score_scale, gpt2_dtype dtype, gpt2_stream_t stream) {
  if (!valid_dtype(dtype) || B < 0 || T < 0 || n_head <= 0 || head_dim <= 0) return GPT2_ERR_ARG;
  if (!(score_scale > 0.f) || !std::isfinite(score_scale)) return GPT2_ERR_ARG;
  if (head_dim != 64 || !is16(dtype)) return GPT2_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * n_head > INT_MAX || T > 65535 * 64) return GPT2_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return GPT2_OK;
  if (!qkv || !out || !lse || !aligned16(qkv) || !aligned16(out)) return GPT2_ERR_ARG;
  const double pairs = static_cast<double>(B) * n_head * T * (T + 1.0) / 2.0;
  ProfScope prof(dtype == GPT2_BF16 ? "attn_causal_bf16_tc" : "attn_causal_f16_tc", 4.0 * 64.0 * pairs,
                 static_cast<double>(B) * T * 4.0 * 64.0 * n_head * 2.0, cs(stream));
  return cuda_status(launch_attention_tc(dtype, qkv, out, B, T, n_head, score_scale, cs(stream), lse));
}

size_t gpt2_attention_backward_workspace_bytes(int B, int T, int n_head) {
  if (B < 0 || T < 0 || n_head <= 0) return 0;
  return align256(static_cast<size_t>(B) * n_head * T * 4);
}

int gpt2_attention_causal_backward(const void* qkv, const void* out, const float* lse, const void* dout, void* dqkv,
                                   int B, int T, int n_head, int head_dim, float score_scale, void* ws,
                                   size_t ws_bytes, gpt2_dtype dtype, gpt2_stream_t stream) {
  if (!valid_dtype(dtype) || B < 0 || T < 0 || n_head <= 0 || head_dim <= 0) return GPT2_ERR_ARG;
  if (!(score_scale > 0.f) || !std::isfinite(score_scale)) return GPT2_ERR_ARG;
  if (head_dim != 64 || !is16(dtype)) return GPT2_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * n_head * ((T + 127) / 128) > INT_MAX || static_cast<int64_t>(B) * T > INT_MAX)
    return GPT2_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return GPT2_OK;
  const void* ps[5] = {qkv, out, lse, dout, dqkv};
  for (const void* p : ps)
    if (!p || !aligned16(p)) return GPT2_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return GPT2_ERR_ARG;
  if (ws_bytes < gpt2_attention_backward_workspace_bytes(B, T, n_head)) return GPT2_ERR_WORKSPACE;
  const double pairs = static_cast<double>(B) * n_head * T * (T + 1.0) / 2.0;
  ProfScope prof(dtype == GPT2_BF16 ? "attn_causal_bwd_bf16_tc" : "attn_causal_bwd_f16_tc", 10.0 * 64.0 * pairs,
                 static_cast<double>(B) * T * 64.0 * n_head * 2.0 * 8.0, cs(stream));
  return cuda_status(launch_attention_backward_tc(dtype, qkv, out, lse, dout, dqkv, static_cast<float*>(ws), B, T,
                                                  n_head, score_scale, cs(stream)));
}

size_t gpt2_mlp_workspace_bytes(int64_t M, int F, gpt2_dtype dtype) {
  if (M < 0 || F <= 0 || !valid_dtype(dtype)) return 0;
  return align256(static_cast<size_t>(M) * F * esize(dtype));
}

int gpt2_mlp(const void* x, const void* w_fc, const void* b_fc, const void* w_proj, const void* b_proj,
             const float* residual, float* out, int64_t M, int D, int F, void* ws, size_t ws_bytes,
             gpt2_dtype dtype, gpt2_stream_t stream) {
  if (!valid_dtype(dtype) || M < 0 || M > INT_MAX || D <= 0 || F <= 0) return GPT2_ERR_ARG;
  if (D % 64 != 0 || F % 64 != 0) return GPT2_ERR_UNSUPPORTED;
  if (M == 0) return GPT2_OK;
  const void* ps[6] = {x, w_fc, b_fc, w_proj, b_proj, out};
  for (const void* p : ps)
    if (!p || !aligned16(p)) return GPT2_ERR_ARG;
  if (residual && !aligned16(residual)) return GPT2_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return GPT2_ERR_ARG;
  if (ws_bytes < gpt2_mlp_workspace_bytes(M, F, dtype)) return GPT2_ERR_WORKSPACE;
  return cuda_status(launch_mlp(dtype, x, w_fc, b_fc, w_proj, b_proj, residual, out, M, D, F, ws, cs(stream)));
}

size_t gpt2_workspace_bytes(const gpt2_dims* dims, int B, int T) {
  if (check_dims(dims, false) != GPT2_OK || B < 0 || T < 0) return 0;
  return acts_bytes(dims, static_cast<int64_t>(B) * T);
}

int gpt2_block_forward(const gpt2_dims* dims, const gpt2_block_weights* w, const float* x_in, float* x_out, int B,
                       int T, void* ws, size_t ws_bytes, gpt2_stream_t stream) {
  return gpt2_block_forward_layer(dims, w, 0, x_in, x_out, B, T, ws, ws_bytes, stream);
}

int gpt2_block_forward_layer(const gpt2_dims* dims, const gpt2_block_weights* w, int layer, const float* x_in,
                             float* x_out, int B, int T, void* ws, size_t ws_bytes, gpt2_stream_t stream) {
  GPT2_TRY(check_dims(dims, false));
  if (layer < 0) return GPT2_ERR_ARG;
  GPT2_TRY(check_block_ptrs(w));
  if (B < 0 || T < 0 || static_cast<int64_t>(B) * T > INT_MAX) return GPT2_ERR_ARG;
  if (B == 0 || T == 0) return GPT2_OK;
  if (!x_in || !x_out || !aligned16(x_in) || !aligned16(x_out)) return GPT2_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return GPT2_ERR_ARG;
  if (ws_bytes < gpt2_workspace_bytes(dims, B, T)) return GPT2_ERR_WORKSPACE;
  const int64_t M = static_cast<int64_t>(B) * T;
  Acts A = carve_acts(ws, dims, M);
  cudaStream_t s = cs(stream);
  GPT2_CUDA(layernorm(x_in, w->ln1_g, w->ln1_b, A.a, M, dims->d_model, dims->eps, GPT2_F32, dims->dtype, s));
  return block_body(dims, w, layer, x_in, x_out, B, T, A, s);
}

size_t gpt2_block_backward_workspace_bytes(const gpt2_dims* dims, int B, int T) {
  if (check_dims(dims, false) != GPT2_OK || dims->dtype != GPT2_F32 || B < 0 || T < 0) return 0;
  return bwd_ws_bytes(dims, B, T);
}

int gpt2_block_backward(const gpt2_dims* dims, const gpt2_block_weights* w, int layer, const float* x_in,
                        const float* dx_out, float* dx_in, const gpt2_block_grads* grads, int B, int T, void* ws,
                        size_t ws_bytes, gpt2_stream_t stream) {
  GPT2_TRY(check_dims(dims, false));
  GPT2_TRY(check_block_ptrs(w));
  if (dims->dtype != GPT2_F32) return GPT2_ERR_UNSUPPORTED;
  if (layer < 0 || B < 0 || T < 0 || static_cast<int64_t>(B) * T > INT_MAX) return GPT2_ERR_ARG;
  if (T > 4096 || B > 65535) return GPT2_ERR_UNSUPPORTED;  // the attention kernels' grid holds B in y
  if (B == 0 || T == 0) return GPT2_OK;
  if (!grads || !x_in || !dx_out || !dx_in) return GPT2_ERR_ARG;
  const void* gs[12] = {grads->ln1_g, grads->ln1_b, grads->w_qkv, grads->b_qkv, grads->w_o,    grads->b_o,
                        grads->ln2_g, grads->ln2_b, grads->w_fc,  grads->b_fc,  grads->w_proj, grads->b_proj};
  for (const void* p : gs)
    if (!p || !aligned16(p)) return GPT2_ERR_ARG;
  if (!aligned16(x_in) || !aligned16(dx_out) || !aligned16(dx_in)) return GPT2_ERR_ARG;
  const int64_t M = static_cast<int64_t>(B) * T;
  const int D = dims->d_model;
  const size_t bytes = static_cast<size_t>(M) * D * 4;
  auto overlap = [&](const void* a, const void* b) {
    const char* x = static_cast<const char*>(a);
    const char* y = static_cast<const char*>(b);
    return x < y + bytes && y < x + bytes;
  };
  if (overlap(dx_in, x_in) || overlap(dx_in, dx_out)) return GPT2_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return GPT2_ERR_ARG;
  if (ws_bytes < bwd_ws_bytes(dims, B, T)) return GPT2_ERR_WORKSPACE;
  return block_backward_f32(dims, w, layer, x_in, dx_out, dx_in, grads, B, T, ws, cs(stream));
}

int gpt2_forward_logits(const gpt2_dims* dims, const gpt2_model_weights* w, const int32_t* tokens, void* logits,
                        int64_t ld, gpt2_dtype logits_t, int B, int T, void* ws, size_t ws_bytes,
                        gpt2_stream_t stream) {
  GPT2_TRY(check_model(dims, w));
  if (!valid_dtype(logits_t)) return GPT2_ERR_ARG;
  if (logits_t != GPT2_F32 && logits_t != dims->dtype) return GPT2_ERR_UNSUPPORTED;
  if (B < 0 || T < 0 || static_cast<int64_t>(B) * T > INT_MAX || ld < dims->vocab) return GPT2_ERR_ARG;
  if (T > dims->n_pos) return GPT2_ERR_ARG;
  if (is16(dims->dtype) && (ld * static_cast<int64_t>(esize(logits_t))) % 16 != 0) return GPT2_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return GPT2_OK;
  if (!tokens || !logits || !aligned16(logits)) return GPT2_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return GPT2_ERR_ARG;
  if (ws_bytes < gpt2_workspace_bytes(dims, B, T)) return GPT2_ERR_WORKSPACE;
  const int64_t M = static_cast<int64_t>(B) * T;
  const gpt2_dtype dt = dims->dtype;
  Acts A = carve_acts(ws, dims, M);
  KeyBuilder kb;
  kb.add(1).dims(dims).model(w, dims->n_layer).ptr(tokens).ptr(logits).add(ld).add(logits_t).add(B).add(T).ptr(ws);
  return run_graphed(kb, cs(stream), [&](cudaStream_t s) -> int {
    GPT2_TRY(forward_to_lnf(dims, w, tokens, B, T, A, s));
    GPT2_CUDA(linear(dt, A.a, w->wte, nullptr, nullptr, logits, M, dims->vocab, dims->d_model, ld, true,
                     GPT2_EPI_NONE, logits_t, s));
    return GPT2_OK;
  });
}


size_t gpt2_loss_workspace_bytes(const gpt2_dims* dims, int B, int T) {
  if (check_dims(dims, true) != GPT2_OK || B < 0 || T < 0) return 0;
  const int64_t M = static_cast<int64_t>(B) * T;
  return acts_bytes(dims, M) + loss_extra_bytes(dims, M);
}

int gpt2_forward_loss(const gpt2_dims* dims, const gpt2_model_weights* w, const int32_t* tokens,
                      const int32_t* labels, float* token_loss, float* lse, float* mean_loss, int B, int T, void* ws,
                      size_t ws_bytes, gpt2_stream_t stream) {
  GPT2_TRY(check_model(dims, w));
  if (B < 0 || T < 0 || static_cast<int64_t>(B) * T > INT_MAX) return GPT2_ERR_ARG;
  if (T > dims->n_pos) return GPT2_ERR_ARG;
  if (B == 0) return GPT2_OK;
  if (T < 2 || !tokens) return GPT2_ERR_ARG;
  if (!token_loss && !lse && !mean_loss) return GPT2_ERR_ARG;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return GPT2_ERR_ARG;
  if (ws_bytes < gpt2_loss_workspace_bytes(dims, B, T)) return GPT2_ERR_WORKSPACE;
  const int64_t M = static_cast<int64_t>(B) * T;
  const gpt2_dtype dt = dims->dtype;
  const int D = dims->d_model, V = dims->vocab;
  if (!labels) labels = tokens;
  Acts A = carve_acts(ws, dims, M);
  KeyBuilder kb;
  kb.add(2).dims(dims).model(w, dims->n_layer).ptr(tokens).ptr(labels).ptr(token_loss).ptr(lse).ptr(mean_loss).add(B)
      .add(T).ptr(ws);
  return run_graphed(kb, cs(stream), [&](cudaStream_t s) -> int {
    Carve c(static_cast<char*>(ws) + acts_bytes(dims, M));
    float* tgt = c.take<float>(M, 4);
    float* tl_scratch = c.take<float>(M, 4);
    GPT2_TRY(forward_to_lnf(dims, w, tokens, B, T, A, s));
    float2* part;
    int n_part = 1;
    if (loss_fused(dims, M)) {
      part = c.take<float2>(M * lse_max_partials(V), sizeof(float2));
      const double e = static_cast<double>(esize(dt));
      ProfScope prof(dt == GPT2_BF16 ? "gemm_lse_bf16_tcgen05" : "gemm_lse_f16_tcgen05", 2.0 * M * V * D,
                     (static_cast<double>(M) + V) * D * e, s);
      GPT2_CUDA(launch_gemm_lse_16(dt, A.a, w->wte, M, V, D, labels, T, part, tgt, &n_part, s));
    } else {
      part = c.take<float2>(M, sizeof(float2));
      float* logits = c.take<float>(M * loss_ld(dims), 4);
      GPT2_CUDA(linear(dt, A.a, w->wte, nullptr, nullptr, logits, M, V, D, loss_ld(dims), true, GPT2_EPI_NONE,
                       GPT2_F32, s));
      ProfScope prof("lse_from_logits", 3.0 * M * V, 4.0 * M * V, s);
      GPT2_CUDA(launch_lse_from_logits(logits, loss_ld(dims), M, V, labels, T, part, tgt, s));
    }
    ProfScope prof("loss_reduce", 4.0 * M * n_part, 8.0 * M * n_part + 12.0 * M, s);
    GPT2_CUDA(launch_loss_rows(part, n_part, tgt, labels, B, T, V, lse, token_loss ? token_loss : tl_scratch,
                               mean_loss, s));
    return GPT2_OK;
  });
}

size_t gpt2_train_workspace_bytes(const gpt2_dims* dims, int B, int T) {
  if (check_dims(dims, true) != GPT2_OK || dims->dtype != GPT2_BF16 || B < 0 || T < 0) return 0;
  return carve_train(nullptr, dims, B, T).bytes;
}

int gpt2_forward_backward(const gpt2_dims* dims, const gpt2_model_weights* w, const int32_t* tokens,
                          const int32_t* labels, const gpt2_model_grads* grads, float* mean_loss, int B, int T,
                          void* ws, size_t ws_bytes, gpt2_stream_t stream) {
  GPT2_TRY(check_model(dims, w));
  if (dims->dtype != GPT2_BF16) return GPT2_ERR_UNSUPPORTED;
  GPT2_TRY(check_grads(dims, grads));
  if (B < 0 || T < 0 || static_cast<int64_t>(B) * T > INT_MAX) return GPT2_ERR_ARG;
  if (T > dims->n_pos) return GPT2_ERR_ARG;
  if (B == 0) return GPT2_OK;
  if (T < 2 || !tokens || !mean_loss) return GPT2_ERR_ARG;
  if (static_cast<int64_t>(B) * dims->n_head * ((T + 127) / 128) > INT_MAX) return GPT2_ERR_UNSUPPORTED;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return GPT2_ERR_ARG;
  if (ws_bytes < gpt2_train_workspace_bytes(dims, B, T)) return GPT2_ERR_WORKSPACE;
  TrainBufs t = carve_train(ws, dims, B, T);
  KeyBuilder kb;
  kb.add(3).dims(dims).model(w, dims->n_layer).ptr(tokens).ptr(labels).ptr(mean_loss).add(B).add(T).ptr(ws);
  kb.ptr(grads->wte).ptr(grads->wpe).ptr(grads->lnf_g).ptr(grads->lnf_b);
  for (int l = 0; l < dims->n_layer; ++l) {
    const gpt2_block_grads& g = grads->blocks[l];
    kb.ptr(g.ln1_g).ptr(g.ln1_b).ptr(g.w_qkv).ptr(g.b_qkv).ptr(g.w_o).ptr(g.b_o);
    kb.ptr(g.ln2_g).ptr(g.ln2_b).ptr(g.w_fc).ptr(g.b_fc).ptr(g.w_proj).ptr(g.b_proj);
  }
  return run_graphed(kb, cs(stream), [&](cudaStream_t s) -> int {
    return forward_backward(dims, w, tokens, labels ? labels : tokens, grads, mean_loss, B, T, t, s);
  });
}

size_t gpt2_kv_cache_bytes(const gpt2_dims* dims, int B, int T_max) {
  if (check_dims(dims, true) != GPT2_OK || B < 0 || T_max < 0) return 0;
  return static_cast<size_t>(dims->n_layer) * 2 * B * dims->n_head * static_cast<size_t>(T_max) * 64 *
         esize(dims->dtype);
}

size_t gpt2_decode_workspace_bytes(const gpt2_dims* dims, int B) {
  if (check_dims(dims, true) != GPT2_OK || B < 0) return 0;
  return decode_ws_bytes(dims, B);
}

int gpt2_decode_step(const gpt2_dims* dims, const gpt2_model_weights* w, void* kv_cache, int B, int T_max,
                     int32_t* past_len, const int32_t* tokens, int32_t* next_tokens, float* logits_opt, int64_t ld,
                     void* ws, size_t ws_bytes, gpt2_stream_t stream) {
  GPT2_TRY(check_model(dims, w));
  if (!is16(dims->dtype)) return GPT2_ERR_UNSUPPORTED;
  if (B < 0 || T_max <= 0) return GPT2_ERR_ARG;
  if (B == 0) return GPT2_OK;
  if (2ll * B * dims->n_head * T_max >= (1ll << 31)) return GPT2_ERR_UNSUPPORTED;
  if (!kv_cache || !past_len || !tokens || !next_tokens || !aligned16(kv_cache)) return GPT2_ERR_ARG;
  if (logits_opt && (ld < dims->vocab || !aligned16(logits_opt))) return GPT2_ERR_ARG;
  if (logits_opt && ld % 4 != 0) return GPT2_ERR_UNSUPPORTED;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return GPT2_ERR_ARG;
  if (ws_bytes < decode_ws_bytes(dims, B)) return GPT2_ERR_WORKSPACE;
  char* base = static_cast<char*>(ws);
  KeyBuilder kb;
  kb.add(5).dims(dims).model(w, dims->n_layer).ptr(kv_cache).add(B).add(T_max).ptr(past_len).ptr(tokens)
      .ptr(next_tokens).ptr(logits_opt).add(ld).ptr(ws);
  return run_graphed(kb, cs(stream), [&](cudaStream_t s) -> int {
    DecodeGroup G;
    G.d = dims;
    G.w = w;
    G.kv_cache = kv_cache;
    G.B_cache = B;
    G.T_max = T_max;
    G.b0 = 0;
    G.nb = B;
    G.past_len = past_len;
    G.tokens = tokens;
    G.next_tokens = next_tokens;
    G.logits = logits_opt;
    G.ld = ld;
    G.valid = reinterpret_cast<int*>(base);
    G.carve(base + align256(static_cast<size_t>(B) * 4));
    G.s = s;
    GPT2_CUDA(G.embed());
    for (int l = 0; l < dims->n_layer; ++l) GPT2_CUDA(G.layer(l));
    GPT2_CUDA(G.head());
    return GPT2_OK;
  });
}

size_t gpt2_prefill_workspace_bytes(const gpt2_dims* dims, int B, int T) {
  if (check_dims(dims, true) != GPT2_OK || B < 0 || T < 0) return 0;
  return acts_bytes(dims, static_cast<int64_t>(B) * T) + prefill_extra_bytes(dims, B);
}

int gpt2_prefill(const gpt2_dims* dims, const gpt2_model_weights* w, const int32_t* tokens, int B, int T,
                 void* kv_cache, int T_max, int32_t* past_len, int32_t* next_tokens, float* logits_opt, int64_t ld,
                 void* ws, size_t ws_bytes, gpt2_stream_t stream) {
  GPT2_TRY(check_model(dims, w));
  if (!is16(dims->dtype)) return GPT2_ERR_UNSUPPORTED;
  if (B < 0 || T < 0 || static_cast<int64_t>(B) * T > INT_MAX) return GPT2_ERR_ARG;
  if (B == 0) return GPT2_OK;
  if (T < 1 || T > dims->n_pos || T > T_max) return GPT2_ERR_ARG;
  if (2ll * B * dims->n_head * T_max >= (1ll << 31)) return GPT2_ERR_UNSUPPORTED;
  if (!tokens || !kv_cache || !past_len || !next_tokens || !aligned16(kv_cache)) return GPT2_ERR_ARG;
  if (logits_opt && (ld < dims->vocab || !aligned16(logits_opt))) return GPT2_ERR_ARG;
  if (logits_opt && ld % 4 != 0) return GPT2_ERR_UNSUPPORTED;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return GPT2_ERR_ARG;
  if (ws_bytes < gpt2_prefill_workspace_bytes(dims, B, T)) return GPT2_ERR_WORKSPACE;
  const int64_t M = static_cast<int64_t>(B) * T;
  const gpt2_dtype dt = dims->dtype;
  const int D = dims->d_model, V = dims->vocab;
  cudaStream_t s = cs(stream);
  Acts A = carve_acts(ws, dims, M);
  Carve c(static_cast<char*>(ws) + acts_bytes(dims, M));
  int* valid = c.take<int>(B, 4);
  float* x_last = c.take<float>(static_cast<size_t>(B) * D, 4);
  void* a_last = c.take<char>(static_cast<size_t>(B) * D, 2);
  GPT2_TRY(forward_to_lnf(dims, w, tokens, B, T, A, s, kv_cache, T_max, false));
  {
    ProfScope prof("prefill_last_rows", 0.0, 8.0 * B * D, s);
    GPT2_CUDA(launch_prefill_last_rows(A.x, B, T, D, x_last, valid, past_len, s));
  }
  GPT2_CUDA(layernorm(x_last, w->lnf_g, w->lnf_b, a_last, B, D, dims->eps, GPT2_F32, dt, s));
  if (B <= kMaxRowsGemm) {
    float2* cand = c.take<float2>(static_cast<size_t>(B) * rows_argmax_candidates(V), sizeof(float2));
    const int n_cand = rows_argmax_candidates(V);
    {
      ProfScope prof(dt == GPT2_BF16 ? "gemm_rows_bf16_tcgen05" : "gemm_rows_f16_tcgen05", 2.0 * B * V * D,
                     (static_cast<double>(B) + V) * D * esize(dt) + (logits_opt ? 4.0 * B * V : 0.0), s);
      GPT2_CUDA(launch_gemm_rows_16(dt, a_last, w->wte, nullptr, nullptr, logits_opt, B, V, D, logits_opt ? ld : V,
                                    true, GPT2_EPI_NONE, GPT2_F32, s, cand));
    }
    ProfScope prof("argmax_candidates", static_cast<double>(B) * n_cand, static_cast<double>(B) * n_cand * 8.0, s);
    GPT2_CUDA(launch_argmax_candidates(cand, n_cand, B, valid, next_tokens, nullptr, s));
    return GPT2_OK;
  }
  const int64_t Vp = (static_cast<int64_t>(V) + 3) & ~static_cast<int64_t>(3);
  float* lg = c.take<float>(static_cast<size_t>(B) * Vp, 4);
  float* out = logits_opt ? logits_opt : lg;
  const int64_t lld = logits_opt ? ld : Vp;
  GPT2_CUDA(linear(dt, a_last, w->wte, nullptr, nullptr, out, B, V, D, lld, true, GPT2_EPI_NONE, GPT2_F32, s));
  ProfScope prof("argmax_rows", static_cast<double>(B) * V, static_cast<double>(B) * V * 4.0, s);
  GPT2_CUDA(launch_argmax_rows(out, lld, B, V, valid, next_tokens, nullptr, s));
  return GPT2_OK;
}

int gpt2_profile_begin(int max_launches) {
  if (max_launches <= 0 || max_launches > (1 << 20)) return GPT2_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  g_prof.on = false;
  g_prof.release();
  g_prof.ev.resize(static_cast<size_t>(2) * max_launches);
  for (auto& e : g_prof.ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      g_prof.release();
      return GPT2_ERR_CUDA;
    }
  }
  g_prof.on = true;
  return GPT2_OK;
}

int gpt2_profile_end(void) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  g_prof.on = false;
  return GPT2_OK;
}

int gpt2_profile_read(gpt2_profile_entry* out, int max_entries, int* n_entries) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (g_prof.on || max_entries < 0 || (!out && max_entries > 0)) return GPT2_ERR_ARG;
  const int n = static_cast<int>(g_prof.names.size());
  if (n_entries) *n_entries = n;
  for (int i = 0; i < n && i < max_entries; ++i) {
    std::memset(&out[i], 0, sizeof(out[i]));
    std::strncpy(out[i].name, g_prof.names[i].c_str(), sizeof(out[i].name) - 1);
  }
  for (const ProfRec& r : g_prof.recs) {
    if (cudaEventSynchronize(g_prof.ev[r.ev0 + 1]) != cudaSuccess) return GPT2_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof.ev[r.ev0], g_prof.ev[r.ev0 + 1]) != cudaSuccess) return GPT2_ERR_CUDA;
    if (r.name_id < max_entries) {
      gpt2_profile_entry& e = out[r.name_id];
      e.launches += 1;
      e.ms += ms;
      e.flops += r.flops;
      e.bytes += r.bytes;
    }
  }
  return GPT2_OK;
}

}  // extern "C"
