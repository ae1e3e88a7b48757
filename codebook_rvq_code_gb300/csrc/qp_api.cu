// C ABI of libqp: handle life cycle, weight validation and packing, and the
// argument checks in front of the frame loop.  See include/qp.h.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "qp_internal.h"
#include "../../include/qp_debug.h"
#include "../../include/qp_sched.h"

namespace {

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

bool geometry_supported(const qp_geometry& g) {
  if (g.hidden <= 0 || g.layers <= 0 || g.layers > qp::kMaxLayers) return false;
  if (g.head_dim != qp::kHeadDim) return false;
  if (g.n_kv_heads <= 0 || g.n_q_heads <= 0 || g.n_q_heads % g.n_kv_heads) return false;
  if (g.n_steps < 1 || g.n_steps > qp::kMaxSteps) return false;
  // code tables as wide as the stream (unprojected) or as the Talker state
  // (each step's input then passes through small_to_mtp)
  if (g.code_embed_dim != g.hidden && g.code_embed_dim != g.talker_hidden) return false;
  if (g.hidden % 128 || g.ffn % 128 || g.talker_hidden % 128 || g.vocab % 128) return false;
  if (g.hidden > 4096 || g.vocab > 8192) return false;
  if (g.ffn <= 0 || g.vocab <= 0 || g.talker_hidden <= 0 || g.q0_vocab <= 0) return false;
  if (!(g.rms_eps >= 0.f) || !(g.rope_theta > 0.f)) return false;
  return true;
}

template <typename T>
T* carve(char*& p, size_t count) {
  size_t bytes = (count * sizeof(T) + 255) & ~size_t(255);
  T* r = reinterpret_cast<T*>(p);
  p += bytes;
  return r;
}
template <typename T>
size_t carve_size(size_t count) { return (count * sizeof(T) + 255) & ~size_t(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
// int32 / f32 device arrays are read and written element by element
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

// What a tensor name maps to, and the shape it must have.
struct Slot {
  enum Kind { MATRIX, EMBED, VECTOR } kind;
  int64_t rows, cols;   // cols = 0 for vectors
};

std::unordered_map<std::string, Slot> build_slots(const qp_geometry& g) {
  std::unordered_map<std::string, Slot> m;
  const int64_t d = g.hidden, qw = int64_t(g.n_q_heads) * g.head_dim,
                kvw = int64_t(g.n_kv_heads) * g.head_dim;
  m["code_pred.small_to_mtp_projection.weight"] = {Slot::MATRIX, d, g.talker_hidden};
  m["code_pred.small_to_mtp_projection.bias"] = {Slot::VECTOR, d, 0};
  m["code_pred.output_norm.weight"] = {Slot::VECTOR, d, 0};
  m["talker.codec_embd.weight"] = {Slot::EMBED, g.q0_vocab, g.talker_hidden};
  for (int j = 0; j < g.n_steps; ++j) {
    m["code_pred.codec_embd." + std::to_string(j) + ".weight"] = {Slot::EMBED, g.vocab, g.code_embed_dim};
    m["code_pred.lm_head." + std::to_string(j) + ".weight"] = {Slot::MATRIX, g.vocab, d};
  }
  for (int l = 0; l < g.layers; ++l) {
    std::string p = "code_pred.blk." + std::to_string(l) + ".";
    m[p + "attn_norm.weight"] = {Slot::VECTOR, d, 0};
    m[p + "attn_q.weight"] = {Slot::MATRIX, qw, d};
    m[p + "attn_k.weight"] = {Slot::MATRIX, kvw, d};
    m[p + "attn_v.weight"] = {Slot::MATRIX, kvw, d};
    m[p + "attn_output.weight"] = {Slot::MATRIX, d, qw};
    m[p + "attn_q_norm.weight"] = {Slot::VECTOR, g.head_dim, 0};
    m[p + "attn_k_norm.weight"] = {Slot::VECTOR, g.head_dim, 0};
    m[p + "ffn_norm.weight"] = {Slot::VECTOR, d, 0};
    m[p + "ffn_gate.weight"] = {Slot::MATRIX, g.ffn, d};
    m[p + "ffn_up.weight"] = {Slot::MATRIX, g.ffn, d};
    m[p + "ffn_down.weight"] = {Slot::MATRIX, d, g.ffn};
  }
  return m;
}

// A packed matrix: 16-bit, or Q8_0 (int8 values and f16 scales) plus its
// f16 hi and lo images for the small-batch engine.
size_t matrix_bytes(int fmt, int64_t N, int64_t K) {
  return fmt == qp::WF_BF16 ? carve_size<uint8_t>(size_t(N) * K * 2)
                            : carve_size<uint8_t>(size_t(N) * K) + carve_size<__half>(size_t(N) * (K / 32)) +
                                  2 * carve_size<uint8_t>(size_t(N) * K * 2);
}

// The engine that serves a call (qp_debug.h, qp_engine).
qp_status run(qp_handle* h, const qp::RunArgs& a, cudaStream_t s) {
  if (h->deterministic) {   // the tile engine's deterministic schedule
    if (h->engine == QP_ENGINE_SMALL || h->engine == QP_ENGINE_CLUSTER) return QP_ERR_ARG;
    return qp::run_frames_persistent(h, a, s);
  }
  if (h->engine == QP_ENGINE_CLUSTER || h->engine == QP_ENGINE_AUTO) {
    const bool cl = qp::cluster_supported(h, a);
    if (h->engine == QP_ENGINE_CLUSTER) return cl ? qp::run_frames_cluster(h, a, s) : QP_ERR_ARG;
    if (cl && (!qp::cluster_ext(h) || a.B >= qp::kClusterExtAutoFrames)) return qp::run_frames_cluster(h, a, s);
  }
  const bool sm = qp::small_supported(h, a);
  if (h->engine == QP_ENGINE_SMALL && !sm) return QP_ERR_ARG;
  const bool pick = h->engine == QP_ENGINE_SMALL || (h->engine == QP_ENGINE_AUTO && a.B <= qp::kSmallAutoFrames);
  if (sm && pick) return qp::run_frames_small(h, a, static_cast<uint8_t*>(h->sarena), h->scr, h->max_batch, s);
  return qp::run_frames_persistent(h, a, s);
}

}  // namespace

extern "C" {

int qp_abi_version(void) { return QP_ABI_VERSION; }

const char* qp_status_string(qp_status s) {
  switch (s) {
    case QP_OK: return "ok";
    case QP_ERR_ARG: return "invalid argument";
    case QP_ERR_STATE: return "invalid state (weights not loaded?)";
    case QP_ERR_WEIGHT_MISSING: return "weight tensor missing";
    case QP_ERR_WEIGHT_SHAPE: return "weight tensor has the wrong shape";
    case QP_ERR_WEIGHT_DTYPE: return "weight tensor has an unsupported storage type";
    case QP_ERR_CUDA: return "CUDA runtime error";
    case QP_ERR_TIMEOUT: return "device wait timed out";
    case QP_ERR_BAD_TOKEN: return "token out of range";
    case QP_ERR_OOM: return "device out of memory";
    case QP_ERR_UNKNOWN_WEIGHT: return "unknown weight tensor name";
    case QP_ERR_DUPLICATE_WEIGHT: return "weight tensor supplied twice";
  }
  return "unknown status";
}

qp_status qp_default_geometry(qp_geometry* g) {
  if (!g) return QP_ERR_ARG;
  g->hidden = 1024; g->layers = 5; g->n_q_heads = 16; g->n_kv_heads = 8; g->head_dim = 128;
  g->ffn = 3072; g->vocab = 2048; g->n_steps = 15; g->talker_hidden = 2048;
  g->code_embed_dim = 1024; g->q0_vocab = 2048; g->rms_eps = 1e-6f; g->rope_theta = 1e6f;
  return QP_OK;
}

qp_status qp_create(const qp_geometry* gp, int max_batch, qp_handle** out) {
  if (!out) return QP_ERR_ARG;
  *out = nullptr;
  if (!gp || max_batch < 1 || max_batch > 65536) return QP_ERR_ARG;
  if (!geometry_supported(*gp)) return QP_ERR_ARG;
  const qp_geometry& g = *gp;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QP_ERR_CUDA;
  auto* h = new qp_handle();
  h->g = g;
  h->max_batch = max_batch;
  h->device = dev;
  if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->clock_khz, cudaDevAttrClockRate, dev) != cudaSuccess) {
    delete h;
    return QP_ERR_CUDA;
  }
  // the persistent kernel's scratch, plus its per-call synchronisation region
  h->scr = qp::scratch_layout(g, max_batch);
  if (cudaMalloc(&h->sarena, h->scr.total) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return QP_ERR_OOM;
  }
  h->sarena_bytes = h->scr.total;
  // the cluster engine's scratch, where it serves this geometry
  if (qp::cluster_geometry_ok(g)) {
    h->cmax_batch = std::min(max_batch, qp::kClusterMaxFrames);
    if (cudaMalloc(&h->carena, qp::cluster_scratch_bytes(g, h->cmax_batch)) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(h->sarena);
      delete h;
      return QP_ERR_OOM;
    }
  }
  // small fixed buffers: status word, RoPE table, host-entry staging
  const int ctx = g.n_steps + 1;
  const size_t fbytes = carve_size<int>(64) + carve_size<float2>(size_t(ctx) * 64) +
                        carve_size<float>(size_t(max_batch) * g.talker_hidden) + carve_size<int32_t>(max_batch) +
                        carve_size<int32_t>(size_t(max_batch) * g.n_steps);
  if (cudaMalloc(&h->farena, fbytes) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->sarena);
    if (h->carena) cudaFree(h->carena);
    delete h;
    return QP_ERR_OOM;
  }
  char* p = static_cast<char*>(h->farena);
  h->status = carve<int>(p, 64);
  h->rope_cs = carve<float2>(p, size_t(ctx) * 64);
  h->H_stage = carve<float>(p, size_t(max_batch) * g.talker_hidden);
  h->q0_stage = carve<int32_t>(p, max_batch);
  h->codes_stage = carve<int32_t>(p, size_t(max_batch) * g.n_steps);

  // RoPE table: angle pos * theta^(-2i/head_dim) formed in double, rounded once.
  std::vector<float2> cs(size_t(ctx) * 64);
  for (int pos = 0; pos < ctx; ++pos)
    for (int i = 0; i < 64; ++i) {
      const double ang = pos * std::pow(double(g.rope_theta), -2.0 * i / g.head_dim);
      cs[size_t(pos) * 64 + i] = make_float2(float(std::cos(ang)), float(std::sin(ang)));
    }
  if (cudaMemset(h->sarena, 0, h->scr.total) != cudaSuccess ||
      cudaMemcpy(h->rope_cs, cs.data(), cs.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(h->status, 0, 64 * sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->sarena);
    if (h->carena) cudaFree(h->carena);
    cudaFree(h->farena);
    delete h;
    return QP_ERR_CUDA;
  }
  *out = h;
  return QP_OK;
}

qp_status qp_load_weights(qp_handle* h, const qp_weight* w, int n, qp_stream sv) {
  if (!h || !w || n <= 0) return QP_ERR_ARG;
  DeviceGuard dg(h->device);
  if (!dg.ok) return QP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(sv);
  const qp_geometry& g = h->g;
  auto slots = build_slots(g);
  std::unordered_map<std::string, int> seen;
  // one format for the projection and layer matrices, one for the lm-heads
  // (16-bit sources, f16 or bf16, pack to the same f16 operand format), one
  // 16-bit encoding for all embedding tables
  int fmt = -1, hfmt = -1, efmt = -1;
  for (int i = 0; i < n; ++i) {
    if (!w[i].name) return QP_ERR_ARG;
    auto it = slots.find(w[i].name);
    if (it == slots.end()) return QP_ERR_UNKNOWN_WEIGHT;
    if (seen.count(w[i].name)) return QP_ERR_DUPLICATE_WEIGHT;
    seen[w[i].name] = i;
    const Slot& sl = it->second;
    if (!w[i].dev_ptr) return QP_ERR_ARG;
    if (w[i].shape[0] != sl.rows || w[i].shape[1] != sl.cols) return QP_ERR_WEIGHT_SHAPE;
    if (sl.kind == Slot::VECTOR && w[i].dtype != QP_F32) return QP_ERR_WEIGHT_DTYPE;
    if (sl.kind == Slot::EMBED) {
      if (w[i].dtype != QP_BF16 && w[i].dtype != QP_F16) return QP_ERR_WEIGHT_DTYPE;
      if (efmt >= 0 && int(w[i].dtype) != efmt) return QP_ERR_WEIGHT_DTYPE;   // one encoding for all tables
      efmt = int(w[i].dtype);
    }
    if (sl.kind == Slot::MATRIX) {
      if (w[i].dtype != QP_BF16 && w[i].dtype != QP_F16 && w[i].dtype != QP_Q8_0) return QP_ERR_WEIGHT_DTYPE;
      const int f = w[i].dtype == QP_Q8_0 ? qp::WF_Q8_0 : qp::WF_BF16;
      int& slot_fmt = std::strncmp(w[i].name, "code_pred.lm_head.", 18) == 0 ? hfmt : fmt;
      if (slot_fmt >= 0 && f != slot_fmt) return QP_ERR_WEIGHT_DTYPE;
      slot_fmt = f;
    }
    if ((w[i].dtype == QP_BF16 || w[i].dtype == QP_F16) && !aligned16(w[i].dev_ptr)) return QP_ERR_ARG;
    if (w[i].dtype == QP_F32 && (reinterpret_cast<uintptr_t>(w[i].dev_ptr) & 3)) return QP_ERR_ARG;
  }
  for (auto& kv : slots)
    if (!seen.count(kv.first)) return QP_ERR_WEIGHT_MISSING;
  // 16-bit heads over Q8_0 matrices (the exporter's layout) are served;
  // Q8_0 heads need Q8_0 matrices
  if (hfmt == qp::WF_Q8_0 && fmt != qp::WF_Q8_0) return QP_ERR_WEIGHT_DTYPE;

  const int64_t d = g.hidden, qw = int64_t(g.n_q_heads) * 128, kvw = int64_t(g.n_kv_heads) * 128;
  size_t bytes = matrix_bytes(fmt, d, g.talker_hidden) + carve_size<float>(d) +
                 carve_size<uint16_t>(size_t(g.q0_vocab) * g.talker_hidden) + carve_size<float>(d);
  for (int l = 0; l < g.layers; ++l)
    bytes += matrix_bytes(fmt, qw + 2 * kvw, d) + matrix_bytes(fmt, d, qw) + matrix_bytes(fmt, 2 * g.ffn, d) +
             matrix_bytes(fmt, d, g.ffn) + 2 * carve_size<float>(d) + 2 * carve_size<float>(128);
  for (int j = 0; j < g.n_steps; ++j)
    bytes += carve_size<uint16_t>(size_t(g.vocab) * g.code_embed_dim) + carve_size<float>(g.vocab) +
             matrix_bytes(hfmt, g.vocab, d);

  if (h->warena) {
    cudaDeviceSynchronize();
    cudaFree(h->warena);
    h->warena = nullptr;
    h->loaded = false;
  }
  if (cudaMalloc(&h->warena, bytes) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_OOM;
  }
  h->warena_bytes = bytes;
  h->wfmt = fmt;
  h->hfmt = hfmt;
  h->embed_f16 = efmt == QP_F16;
  char* p = static_cast<char*>(h->warena);
  cudaError_t err = cudaSuccess;
  auto chk = [&](cudaError_t e) { if (e != cudaSuccess && err == cudaSuccess) err = e; };
  auto get = [&](const std::string& name) -> const qp_weight& { return w[seen[name]]; };
  auto alloc_mat = [&](int64_t N, int64_t K, int mfmt) {
    qp::PackedMat m;
    m.N = int(N); m.K = int(K); m.fmt = mfmt;
    if (mfmt == qp::WF_BF16) {
      m.w = carve<uint8_t>(p, size_t(N) * K * 2);
    } else {
      m.w = carve<uint8_t>(p, size_t(N) * K);
      m.scale = carve<__half>(p, size_t(N) * (K / 32));
      m.w16[0] = carve<uint8_t>(p, size_t(N) * K * 2);
      m.w16[1] = carve<uint8_t>(p, size_t(N) * K * 2);
    }
    return m;
  };
  auto put = [&](const qp::PackedMat& m, int row0, const std::string& name) {
    const qp_weight& src = get(name);
    chk(qp::pack_rows(src.dev_ptr, m.fmt, src.dtype == QP_F16, int(src.shape[0]), int(src.shape[1]), m, row0, s));
  };
  auto put_vec = [&](const std::string& name, int64_t count) {
    float* dst = carve<float>(p, count);
    chk(cudaMemcpyAsync(dst, get(name).dev_ptr, size_t(count) * 4, cudaMemcpyDeviceToDevice, s));
    return static_cast<const float*>(dst);
  };

  h->proj = alloc_mat(d, g.talker_hidden, fmt);
  put(h->proj, 0, "code_pred.small_to_mtp_projection.weight");
  h->b_proj = put_vec("code_pred.small_to_mtp_projection.bias", d);
  {
    uint16_t* e0 = carve<uint16_t>(p, size_t(g.q0_vocab) * g.talker_hidden);
    chk(cudaMemcpyAsync(e0, get("talker.codec_embd.weight").dev_ptr, size_t(g.q0_vocab) * g.talker_hidden * 2,
                        cudaMemcpyDeviceToDevice, s));
    h->e0 = e0;
  }
  h->out_norm = put_vec("code_pred.output_norm.weight", d);
  for (int l = 0; l < g.layers; ++l) {
    const std::string pre = "code_pred.blk." + std::to_string(l) + ".";
    qp::LayerW& L = h->layer[l];
    L.qkv = alloc_mat(qw + 2 * kvw, d, fmt);
    put(L.qkv, 0, pre + "attn_q.weight");
    put(L.qkv, int(qw), pre + "attn_k.weight");
    put(L.qkv, int(qw + kvw), pre + "attn_v.weight");
    L.o = alloc_mat(d, qw, fmt);
    put(L.o, 0, pre + "attn_output.weight");
    L.gu = alloc_mat(2 * g.ffn, d, fmt);
    put(L.gu, 0, pre + "ffn_gate.weight");
    put(L.gu, g.ffn, pre + "ffn_up.weight");
    L.down = alloc_mat(d, g.ffn, fmt);
    put(L.down, 0, pre + "ffn_down.weight");
    L.attn_norm = put_vec(pre + "attn_norm.weight", d);
    L.ffn_norm = put_vec(pre + "ffn_norm.weight", d);
    L.q_norm = put_vec(pre + "attn_q_norm.weight", 128);
    L.k_norm = put_vec(pre + "attn_k_norm.weight", 128);
  }
  for (int j = 0; j < g.n_steps; ++j) {
    const size_t ce = size_t(g.code_embed_dim);
    uint16_t* e = carve<uint16_t>(p, size_t(g.vocab) * ce);
    chk(cudaMemcpyAsync(e, get("code_pred.codec_embd." + std::to_string(j) + ".weight").dev_ptr,
                        size_t(g.vocab) * ce * 2, cudaMemcpyDeviceToDevice, s));
    h->embed[j] = e;
    float* ss = carve<float>(p, g.vocab);
    chk(qp::row_sumsq_e16(e, g.vocab, int(ce), h->embed_f16, ss, s));
    h->embed_ss[j] = ss;
    h->head[j] = alloc_mat(g.vocab, d, hfmt);
    put(h->head[j], 0, "code_pred.lm_head." + std::to_string(j) + ".weight");
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  h->loaded = true;
  return QP_OK;
}

static qp_status check_run(qp_handle* h, int B, const float* H, const int32_t* q0, int32_t* out_codes,
                           const qp_sampling* samp, bool device_ptrs) {
  if (!h) return QP_ERR_ARG;
  if (!h->loaded) return QP_ERR_STATE;
  if (B < 1 || B > h->max_batch || !H || !q0 || !out_codes) return QP_ERR_ARG;
  if (device_ptrs && (!aligned16(H) || !aligned4(q0) || !aligned4(out_codes))) return QP_ERR_ARG;
  if (samp) {
    if (!(samp->temperature > 0.f) || !std::isfinite(samp->temperature)) return QP_ERR_ARG;
    if (samp->top_k < 1 || samp->top_k > h->g.vocab || !samp->gumbel || !aligned4(samp->gumbel)) return QP_ERR_ARG;
    if (h->g.vocab > qp::kMaxVocab) return QP_ERR_ARG;
  }
  return QP_OK;
}

qp_status qp_predict_frames_ex(qp_handle* h, int B, const float* H, const int32_t* q0, int32_t* out_codes,
                               float* out_logits, const qp_sampling* samp, const int32_t* forced_codes,
                               qp_stream s) {
  qp_status st = check_run(h, B, H, q0, out_codes, samp, true);
  if (st != QP_OK) return st;
  if ((out_logits && !aligned16(out_logits)) || !aligned4(forced_codes)) return QP_ERR_ARG;
  DeviceGuard dg(h->device);
  if (!dg.ok) return QP_ERR_CUDA;
  qp::RunArgs a;
  a.B = B; a.H = H; a.q0 = q0; a.out_codes = out_codes; a.out_logits = out_logits; a.forced = forced_codes;
  if (samp) { a.temperature = samp->temperature; a.top_k = samp->top_k; a.gumbel = samp->gumbel; }
  return run(h, a, static_cast<cudaStream_t>(s));
}

qp_status qp_predict_frames(qp_handle* h, int B, const float* H, const int32_t* q0, int32_t* out_codes,
                            float* out_logits, qp_stream s) {
  return qp_predict_frames_ex(h, B, H, q0, out_codes, out_logits, nullptr, nullptr, s);
}

qp_status qp_predict_frames_host(qp_handle* h, int B, const float* H_host, const int32_t* q0_host,
                                 int32_t* codes_host, const qp_sampling* samp, qp_stream sv) {
  qp_status st = check_run(h, B, H_host, q0_host, codes_host, samp, false);
  if (st != QP_OK) return st;
  DeviceGuard dg(h->device);
  if (!dg.ok) return QP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(sv);
  const qp_geometry& g = h->g;
  if (cudaMemcpyAsync(h->H_stage, H_host, size_t(B) * g.talker_hidden * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(h->q0_stage, q0_host, size_t(B) * 4, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  qp::RunArgs a;
  a.B = B; a.H = h->H_stage; a.q0 = h->q0_stage; a.out_codes = h->codes_stage;
  if (samp) { a.temperature = samp->temperature; a.top_k = samp->top_k; a.gumbel = samp->gumbel; }
  st = run(h, a, s);
  if (st != QP_OK) return st;
  if (cudaMemcpyAsync(codes_host, h->codes_stage, size_t(B) * g.n_steps * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  return QP_OK;
}

qp_status qp_predict_frames_static(qp_handle* h, int B, const float* H, const int32_t* q0, int32_t* out_codes,
                                   float* out_logits, qp_stream s) {
  qp_status st = check_run(h, B, H, q0, out_codes, nullptr, true);
  if (st != QP_OK) return st;
  if (out_logits && !aligned16(out_logits)) return QP_ERR_ARG;
  DeviceGuard dg(h->device);
  if (!dg.ok) return QP_ERR_CUDA;
  qp::RunArgs a;
  a.B = B; a.H = H; a.q0 = q0; a.out_codes = out_codes; a.out_logits = out_logits;
  return qp::run_frames_static(h, a, static_cast<cudaStream_t>(s));
}

// Slots of one state-slot call: each in [0, max_batch), none repeated.
static bool slots_ok(const qp_handle* h, int B, const int32_t* slots) {
  for (int b = 0; b < B; ++b) {
    if (slots[b] < 0 || slots[b] >= h->max_batch) return false;
    for (int c = 0; c < b; ++c)
      if (slots[c] == slots[b]) return false;
  }
  return true;
}

static qp_status run_slots(qp_handle* h, const qp::SlotArgs& a, qp_stream s) {
  DeviceGuard dg(h->device);
  if (!dg.ok) return QP_ERR_CUDA;
  return qp::run_slots_small(h, a, static_cast<uint8_t*>(h->sarena), h->scr, h->max_batch, static_cast<cudaStream_t>(s));
}

// Sampling parameters of a state-slot call: as for qp_predict_frames_ex,
// with the vocabulary within the sampling pass's key array.
static bool slot_sampling_ok(const qp_handle* h, const qp_sampling* samp, qp::SlotArgs& a) {
  if (!samp) return true;
  if (!(samp->temperature > 0.f) || !std::isfinite(samp->temperature)) return false;
  if (samp->top_k < 1 || samp->top_k > h->g.vocab || !samp->gumbel || !aligned4(samp->gumbel)) return false;
  if (h->g.vocab > qp::kMaxVocab) return false;
  a.temperature = samp->temperature; a.top_k = samp->top_k; a.gumbel = samp->gumbel;
  return true;
}

qp_status qp_begin_frames(qp_handle* h, int B, const int32_t* slots, const float* H, const int32_t* q0,
                          int32_t* out_q1, float* out_logits, qp_stream s) {
  return qp_begin_frames_ex(h, B, slots, H, q0, out_q1, out_logits, nullptr, s);
}

qp_status qp_step_frames(qp_handle* h, int B, const int32_t* slots, const int32_t* steps, const int32_t* codes_in,
                         int32_t* out_codes, float* out_logits, qp_stream s) {
  return qp_step_frames_ex(h, B, slots, steps, codes_in, out_codes, out_logits, nullptr, s);
}

qp_status qp_begin_frames_ex(qp_handle* h, int B, const int32_t* slots, const float* H, const int32_t* q0,
                             int32_t* out_q1, float* out_logits, const qp_sampling* samp, qp_stream s) {
  if (!h) return QP_ERR_ARG;
  if (!h->loaded) return QP_ERR_STATE;
  if (B < 1 || B > h->max_batch || B > qp::kSmallMaxFrames || !slots || !H || !q0 || !out_q1) return QP_ERR_ARG;
  if (!aligned16(H) || !aligned4(q0) || !aligned4(out_q1) || (out_logits && !aligned16(out_logits)) ||
      !slots_ok(h, B, slots))
    return QP_ERR_ARG;
  qp::SlotArgs a;
  a.mode = 1; a.B = B; a.slots = slots; a.H = H; a.q0 = q0; a.out_codes = out_q1; a.out_logits = out_logits;
  if (!slot_sampling_ok(h, samp, a)) return QP_ERR_ARG;
  return run_slots(h, a, s);
}

qp_status qp_step_frames_ex(qp_handle* h, int B, const int32_t* slots, const int32_t* steps, const int32_t* codes_in,
                            int32_t* out_codes, float* out_logits, const qp_sampling* samp, qp_stream s) {
  if (!h) return QP_ERR_ARG;
  if (!h->loaded) return QP_ERR_STATE;
  if (B < 1 || B > h->max_batch || B > qp::kSmallMaxFrames || !slots || !steps || !codes_in || !out_codes)
    return QP_ERR_ARG;
  if (!aligned4(codes_in) || !aligned4(out_codes) || (out_logits && !aligned16(out_logits)) || !slots_ok(h, B, slots))
    return QP_ERR_ARG;
  for (int b = 0; b < B; ++b)
    if (steps[b] < 2 || steps[b] > h->g.n_steps) return QP_ERR_ARG;
  qp::SlotArgs a;
  a.mode = 2; a.B = B; a.slots = slots; a.steps = steps; a.codes_in = codes_in; a.out_codes = out_codes;
  a.out_logits = out_logits;
  if (!slot_sampling_ok(h, samp, a)) return QP_ERR_ARG;
  return run_slots(h, a, s);
}

qp_status qp_get_device_status(qp_handle* h, qp_stream sv) {
  if (!h) return QP_ERR_ARG;
  DeviceGuard dg(h->device);
  if (!dg.ok) return QP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(sv);
  int v = 0;
  if (cudaMemcpyAsync(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(h->status, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  return static_cast<qp_status>(v);
}

int qp_launches_per_call(qp_handle* h, int B, int /*sampling*/) {
  if (!h || B < 1 || B > h->max_batch) return -1;
  return 1;   // one persistent kernel per call
}

qp_status qp_set_deterministic(qp_handle* h, int on) {
  if (!h) return QP_ERR_ARG;
  h->deterministic = on != 0;
  return QP_OK;
}

qp_status qp_debug_waits(qp_handle* h, int wait_limit_us, int withhold_gemm) {
  if (!h || wait_limit_us < 0 || withhold_gemm < -1) return QP_ERR_ARG;
  h->wait_ticks = (long long)wait_limit_us * (h->clock_khz > 0 ? h->clock_khz : 2000000) / 1000;
  h->withhold_gemm = withhold_gemm;
  return QP_OK;
}

qp_status qp_set_engine(qp_handle* h, int engine) {
  if (!h || engine < QP_ENGINE_AUTO || engine > QP_ENGINE_CLUSTER) return QP_ERR_ARG;
  h->engine = engine;
  return QP_OK;
}

qp_status qp_trace_enable(qp_handle* h, int enable) {
  if (!h) return QP_ERR_ARG;
#ifndef QP_TRACE
  if (enable) return QP_ERR_STATE;   // the kernels were built without the trace hooks
#endif
  DeviceGuard dg(h->device);
  if (!dg.ok) return QP_ERR_CUDA;
  cudaDeviceSynchronize();
  if (h->trace) {
    cudaFree(h->trace);
    h->trace = nullptr;
    h->trace_phases = 0;
  }
  if (!enable) return QP_OK;
  const int phases = 8192;
  // section stamps [phases][cta][2], then a 16384-word event log per CTA
  const size_t bytes = (size_t(phases) * h->num_sms * 2 + size_t(h->num_sms) * 16384) * sizeof(unsigned long long);
  if (cudaMalloc(&h->trace, bytes) != cudaSuccess) {
    cudaGetLastError();
    h->trace = nullptr;
    return QP_ERR_OOM;
  }
  cudaMemset(h->trace, 0, bytes);
  h->trace_phases = phases;
  return QP_OK;
}

int qp_trace_read(qp_handle* h, uint64_t* host, int phases, int* n_cta) {
  if (!h || !host || phases < 0 || !h->trace) return -1;
  DeviceGuard dg(h->device);
  if (!dg.ok) return -1;
  if (phases > h->trace_phases) phases = h->trace_phases;
  if (n_cta) *n_cta = h->num_sms;
  size_t words = size_t(phases) * h->num_sms * 2;
  if (phases == h->trace_phases) words += size_t(h->num_sms) * 16384;   // and the event logs
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(host, h->trace, words * sizeof(uint64_t), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return phases;
}

qp_status qp_code_embeddings(qp_handle* h, int B, const int32_t* codes, float* out, qp_stream sv) {
  if (!h) return QP_ERR_ARG;
  if (!h->loaded) return QP_ERR_STATE;
  if (B < 0) return QP_ERR_ARG;
  if (B == 0) return QP_OK;
  if (!codes || !out || !aligned16(out) || (reinterpret_cast<uintptr_t>(codes) & 3)) return QP_ERR_ARG;
  DeviceGuard dg(h->device);
  if (!dg.ok) return QP_ERR_CUDA;
  const qp_geometry& g = h->g;
  if (qp::code_embeddings(h->embed, g.n_steps, g.vocab, g.code_embed_dim, codes, B, out, h->status, h->embed_f16,
                          static_cast<cudaStream_t>(sv)) != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  return QP_OK;
}

void qp_destroy(qp_handle* h) {
  if (!h) return;
  {
    DeviceGuard dg(h->device);
    cudaDeviceSynchronize();
    if (h->trace) cudaFree(h->trace);
    if (h->warena) cudaFree(h->warena);
    if (h->sarena) cudaFree(h->sarena);
    if (h->carena) cudaFree(h->carena);
    if (h->farena) cudaFree(h->farena);
  }
  delete h;
}

}  // extern "C"
