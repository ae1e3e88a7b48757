// C ABI of libqp: handle life cycle, weight validation and repacking, and the
// argument checks in front of the frame loop.  See include/qp.h.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include "qp_internal.h"

using qp::QMat;

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
  if (g.code_embed_dim != g.hidden) return false;
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

// What a tensor name maps to, and the shape it must have.
struct Slot {
  enum Kind { MATRIX, EMBED, VECTOR } kind;
  int64_t rows, cols;   // cols = 0 for vectors
  int role;             // see Role
  int layer, index;
};
enum Role {
  R_PROJ_W, R_PROJ_B, R_OUT_NORM, R_E0, R_EMBED, R_HEAD,
  R_ATTN_NORM, R_Q, R_K, R_V, R_O, R_QN, R_KN, R_FFN_NORM, R_GATE, R_UP, R_DOWN
};

std::unordered_map<std::string, Slot> build_slots(const qp_geometry& g) {
  std::unordered_map<std::string, Slot> m;
  const int64_t d = g.hidden, qw = int64_t(g.n_q_heads) * g.head_dim,
                kvw = int64_t(g.n_kv_heads) * g.head_dim;
  m["code_pred.small_to_mtp_projection.weight"] = {Slot::MATRIX, d, g.talker_hidden, R_PROJ_W, -1, -1};
  m["code_pred.small_to_mtp_projection.bias"] = {Slot::VECTOR, d, 0, R_PROJ_B, -1, -1};
  m["code_pred.output_norm.weight"] = {Slot::VECTOR, d, 0, R_OUT_NORM, -1, -1};
  m["talker.codec_embd.weight"] = {Slot::EMBED, g.q0_vocab, g.talker_hidden, R_E0, -1, -1};
  for (int j = 0; j < g.n_steps; ++j) {
    m["code_pred.codec_embd." + std::to_string(j) + ".weight"] = {Slot::EMBED, g.vocab, g.code_embed_dim, R_EMBED, -1, j};
    m["code_pred.lm_head." + std::to_string(j) + ".weight"] = {Slot::MATRIX, g.vocab, d, R_HEAD, -1, j};
  }
  for (int l = 0; l < g.layers; ++l) {
    std::string p = "code_pred.blk." + std::to_string(l) + ".";
    m[p + "attn_norm.weight"] = {Slot::VECTOR, d, 0, R_ATTN_NORM, l, -1};
    m[p + "attn_q.weight"] = {Slot::MATRIX, qw, d, R_Q, l, -1};
    m[p + "attn_k.weight"] = {Slot::MATRIX, kvw, d, R_K, l, -1};
    m[p + "attn_v.weight"] = {Slot::MATRIX, kvw, d, R_V, l, -1};
    m[p + "attn_output.weight"] = {Slot::MATRIX, d, qw, R_O, l, -1};
    m[p + "attn_q_norm.weight"] = {Slot::VECTOR, g.head_dim, 0, R_QN, l, -1};
    m[p + "attn_k_norm.weight"] = {Slot::VECTOR, g.head_dim, 0, R_KN, l, -1};
    m[p + "ffn_norm.weight"] = {Slot::VECTOR, d, 0, R_FFN_NORM, l, -1};
    m[p + "ffn_gate.weight"] = {Slot::MATRIX, g.ffn, d, R_GATE, l, -1};
    m[p + "ffn_up.weight"] = {Slot::MATRIX, g.ffn, d, R_UP, l, -1};
    m[p + "ffn_down.weight"] = {Slot::MATRIX, d, g.ffn, R_DOWN, l, -1};
  }
  return m;
}

size_t matrix_bytes(int fmt, int64_t N, int64_t K) {
  if (fmt == qp::WF_BF16) return carve_size<uint16_t>(size_t(N) * K);
  return carve_size<int8_t>(size_t(N) * K) + carve_size<__half>(size_t(N) * (K / 32));
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
    case QP_ERR_TIMEOUT: return "device barrier timed out";
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
  if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    delete h;
    return QP_ERR_CUDA;
  }
  const size_t R = size_t(2) * max_batch;
  const int qw = g.n_q_heads * g.head_dim, kvw = g.n_kv_heads * g.head_dim;
  int aw = g.hidden;
  if (qw > aw) aw = qw;
  if (g.ffn > aw) aw = g.ffn;
  if (g.talker_hidden > aw) aw = g.talker_hidden;
  h->act_width = aw;
  const int ctx = g.n_steps + 1;
  size_t bytes = 0;
  bytes += carve_size<float>(R * g.hidden);
  bytes += carve_size<uint16_t>(R * aw);
  bytes += carve_size<float>(R * (qw + 2 * kvw));
  bytes += carve_size<float>(R * 2 * g.ffn);
  bytes += carve_size<float>(size_t(g.layers) * max_batch * ctx * 2 * kvw);
  bytes += carve_size<float>(size_t(max_batch) * g.vocab);
  bytes += carve_size<int>(64);
  bytes += carve_size<float2>(size_t(ctx) * (g.head_dim / 2));
  bytes += carve_size<float>(size_t(max_batch) * g.talker_hidden);
  bytes += carve_size<int32_t>(max_batch);
  bytes += carve_size<int32_t>(size_t(max_batch) * g.n_steps);
  const size_t Rpad = (R + 127) / 128 * 128;
  bytes += carve_size<uint16_t>(Rpad * aw);
  bytes += carve_size<unsigned int>(64);
  if (cudaMalloc(&h->sarena, bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return QP_ERR_OOM;
  }
  h->sarena_bytes = bytes;
  char* p = static_cast<char*>(h->sarena);
  h->X = carve<float>(p, R * g.hidden);
  h->act = carve<uint16_t>(p, R * aw);
  h->qkv = carve<float>(p, R * (qw + 2 * kvw));
  h->gu = carve<float>(p, R * 2 * g.ffn);
  h->kv = carve<float>(p, size_t(g.layers) * max_batch * ctx * 2 * kvw);
  h->logits = carve<float>(p, size_t(max_batch) * g.vocab);
  h->status = carve<int>(p, 64);
  h->rope_cs = carve<float2>(p, size_t(ctx) * (g.head_dim / 2));
  h->H_stage = carve<float>(p, size_t(max_batch) * g.talker_hidden);
  h->q0_stage = carve<int32_t>(p, max_batch);
  h->codes_stage = carve<int32_t>(p, size_t(max_batch) * g.n_steps);
  h->pact = carve<uint16_t>(p, Rpad * aw);
  h->sync_words = carve<unsigned int>(p, 64);

  // RoPE table: angle p * theta^(-2i/head_dim) formed in double, rounded once.
  std::vector<float2> cs(size_t(ctx) * (g.head_dim / 2));
  for (int pos = 0; pos < ctx; ++pos)
    for (int i = 0; i < g.head_dim / 2; ++i) {
      double ang = pos * std::pow(double(g.rope_theta), -2.0 * i / g.head_dim);
      cs[size_t(pos) * (g.head_dim / 2) + i] = make_float2(float(std::cos(ang)), float(std::sin(ang)));
    }
  if (cudaMemcpy(h->rope_cs, cs.data(), cs.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(h->status, 0, 64 * sizeof(int)) != cudaSuccess ||
      cudaMemset(h->pact, 0, Rpad * aw * sizeof(uint16_t)) != cudaSuccess ||
      cudaMemset(h->sync_words, 0, 64 * sizeof(unsigned int)) != cudaSuccess) {
    cudaFree(h->sarena);
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
  int fmt = -1;
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
    if (sl.kind == Slot::EMBED && w[i].dtype != QP_BF16) return QP_ERR_WEIGHT_DTYPE;
    if (sl.kind == Slot::MATRIX) {
      if (w[i].dtype != QP_BF16 && w[i].dtype != QP_Q8_0) return QP_ERR_WEIGHT_DTYPE;
      int f = w[i].dtype == QP_BF16 ? qp::WF_BF16 : qp::WF_Q8_0;
      if (fmt >= 0 && f != fmt) return QP_ERR_WEIGHT_DTYPE;   // one format for all matrices
      fmt = f;
    }
  }
  for (auto& kv : slots)
    if (!seen.count(kv.first)) return QP_ERR_WEIGHT_MISSING;

  // Size the arena.
  const int64_t d = g.hidden, qw = int64_t(g.n_q_heads) * g.head_dim, kvw = int64_t(g.n_kv_heads) * g.head_dim;
  size_t bytes = matrix_bytes(fmt, d, g.talker_hidden) + carve_size<float>(d) +
                 carve_size<uint16_t>(size_t(g.q0_vocab) * g.talker_hidden) + carve_size<float>(d);
  for (int l = 0; l < g.layers; ++l)
    bytes += matrix_bytes(fmt, qw + 2 * kvw, d) + matrix_bytes(fmt, d, qw) + matrix_bytes(fmt, 2 * g.ffn, d) +
             matrix_bytes(fmt, d, g.ffn) + 2 * carve_size<float>(d) + 2 * carve_size<float>(g.head_dim);
  for (int j = 0; j < g.n_steps; ++j)
    bytes += carve_size<uint16_t>(size_t(g.vocab) * d) + matrix_bytes(fmt, g.vocab, d);
  // packed copies for the tensor-core engine
  auto pk = [&](int64_t N, int64_t K) { return matrix_bytes(fmt, N, K); };
  bytes += pk(d, g.talker_hidden);
  for (int l = 0; l < g.layers; ++l) bytes += pk(qw + 2 * kvw, d) + pk(d, qw) + pk(2 * g.ffn, d) + pk(d, g.ffn);
  for (int j = 0; j < g.n_steps; ++j) bytes += pk(g.vocab, d);

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
  char* p = static_cast<char*>(h->warena);

  auto alloc_mat = [&](int64_t N, int64_t K) {
    QMat m;
    m.N = int(N); m.K = int(K); m.fmt = fmt;
    if (fmt == qp::WF_BF16) {
      m.w = carve<uint16_t>(p, size_t(N) * K);
    } else {
      m.w = carve<int8_t>(p, size_t(N) * K);
      m.scale = carve<__half>(p, size_t(N) * (K / 32));
    }
    return m;
  };
  // Copy rows [row0, row0 + rows) of matrix m from a caller tensor.
  auto put_rows = [&](const QMat& m, int64_t row0, const qp_weight& src) -> cudaError_t {
    const int64_t rows = src.shape[0], K = src.shape[1];
    if (fmt == qp::WF_BF16) {
      return cudaMemcpyAsync(static_cast<uint16_t*>(const_cast<void*>(m.w)) + row0 * K, src.dev_ptr,
                             size_t(rows) * K * 2, cudaMemcpyDeviceToDevice, s);
    }
    return qp::repack_q8_0(static_cast<const uint8_t*>(src.dev_ptr), int(rows), int(K),
                           static_cast<int8_t*>(const_cast<void*>(m.w)) + row0 * K,
                           const_cast<__half*>(m.scale) + row0 * (K / 32), s);
  };
  auto get = [&](const std::string& name) -> const qp_weight& { return w[seen[name]]; };
  cudaError_t err = cudaSuccess;
  auto chk = [&](cudaError_t e) { if (e != cudaSuccess && err == cudaSuccess) err = e; };
  auto put_vec = [&](const std::string& name, int64_t count) {
    float* dst = carve<float>(p, count);
    chk(cudaMemcpyAsync(dst, get(name).dev_ptr, size_t(count) * 4, cudaMemcpyDeviceToDevice, s));
    return static_cast<const float*>(dst);
  };

  h->proj = alloc_mat(d, g.talker_hidden);
  chk(put_rows(h->proj, 0, get("code_pred.small_to_mtp_projection.weight")));
  h->b_proj = put_vec("code_pred.small_to_mtp_projection.bias", d);
  {
    uint16_t* e0 = carve<uint16_t>(p, size_t(g.q0_vocab) * g.talker_hidden);
    chk(cudaMemcpyAsync(e0, get("talker.codec_embd.weight").dev_ptr, size_t(g.q0_vocab) * g.talker_hidden * 2,
                        cudaMemcpyDeviceToDevice, s));
    h->e0 = e0;
  }
  h->out_norm = put_vec("code_pred.output_norm.weight", d);
  for (int l = 0; l < g.layers; ++l) {
    std::string pre = "code_pred.blk." + std::to_string(l) + ".";
    qp::LayerW& L = h->layer[l];
    L.qkv = alloc_mat(qw + 2 * kvw, d);
    chk(put_rows(L.qkv, 0, get(pre + "attn_q.weight")));
    chk(put_rows(L.qkv, qw, get(pre + "attn_k.weight")));
    chk(put_rows(L.qkv, qw + kvw, get(pre + "attn_v.weight")));
    L.o = alloc_mat(d, qw);
    chk(put_rows(L.o, 0, get(pre + "attn_output.weight")));
    L.gu = alloc_mat(2 * g.ffn, d);
    chk(put_rows(L.gu, 0, get(pre + "ffn_gate.weight")));
    chk(put_rows(L.gu, g.ffn, get(pre + "ffn_up.weight")));
    L.down = alloc_mat(d, g.ffn);
    chk(put_rows(L.down, 0, get(pre + "ffn_down.weight")));
    L.attn_norm = put_vec(pre + "attn_norm.weight", d);
    L.ffn_norm = put_vec(pre + "ffn_norm.weight", d);
    L.q_norm = put_vec(pre + "attn_q_norm.weight", g.head_dim);
    L.k_norm = put_vec(pre + "attn_k_norm.weight", g.head_dim);
  }
  for (int j = 0; j < g.n_steps; ++j) {
    uint16_t* e = carve<uint16_t>(p, size_t(g.vocab) * d);
    chk(cudaMemcpyAsync(e, get("code_pred.codec_embd." + std::to_string(j) + ".weight").dev_ptr,
                        size_t(g.vocab) * d * 2, cudaMemcpyDeviceToDevice, s));
    h->embed[j] = e;
    h->head[j] = alloc_mat(g.vocab, d);
    chk(put_rows(h->head[j], 0, get("code_pred.lm_head." + std::to_string(j) + ".weight")));
  }
  auto pack = [&](const QMat& m) {
    qp::PackedMat pm;
    if (fmt == qp::WF_BF16) {
      pm.w = carve<uint8_t>(p, size_t(m.N) * m.K * 2);
    } else {
      pm.w = carve<uint8_t>(p, size_t(m.N) * m.K);
      pm.scale = carve<__half>(p, size_t(m.N) * (m.K / 32));
    }
    chk(qp::pack_matrix(m, pm, s));
    return pm;
  };
  h->pproj = pack(h->proj);
  for (int l = 0; l < g.layers; ++l) {
    h->player[l].qkv = pack(h->layer[l].qkv);
    h->player[l].o = pack(h->layer[l].o);
    h->player[l].gu = pack(h->layer[l].gu);
    h->player[l].down = pack(h->layer[l].down);
  }
  for (int j = 0; j < g.n_steps; ++j) h->phead[j] = pack(h->head[j]);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return QP_ERR_CUDA;
  }
  h->loaded = true;
  return QP_OK;
}

static qp_status check_run(qp_handle* h, int B, const float* H, const int32_t* q0, int32_t* out_codes,
                           const qp_sampling* samp) {
  if (!h) return QP_ERR_ARG;
  if (!h->loaded) return QP_ERR_STATE;
  if (B < 1 || B > h->max_batch || !H || !q0 || !out_codes) return QP_ERR_ARG;
  if (samp) {
    if (!(samp->temperature > 0.f) || !std::isfinite(samp->temperature)) return QP_ERR_ARG;
    if (samp->top_k < 1 || samp->top_k > h->g.vocab || !samp->gumbel) return QP_ERR_ARG;
  }
  return QP_OK;
}

// The persistent tensor-core engine runs every call; QP_ENGINE=layers selects
// the per-operation kernels (kept while the persistent engine is brought up).
static qp_status dispatch(qp_handle* h, const qp::RunArgs& a, cudaStream_t s) {
  static const char* eng = std::getenv("QP_ENGINE");
  if (eng && std::strcmp(eng, "layers") == 0) return qp::run_frames(h, a, s);
  return qp::run_frames_persistent(h, a, s);
}

qp_status qp_predict_frames_ex(qp_handle* h, int B, const float* H, const int32_t* q0, int32_t* out_codes,
                               float* out_logits, const qp_sampling* samp, const int32_t* forced_codes,
                               qp_stream s) {
  qp_status st = check_run(h, B, H, q0, out_codes, samp);
  if (st != QP_OK) return st;
  DeviceGuard dg(h->device);
  if (!dg.ok) return QP_ERR_CUDA;
  qp::RunArgs a;
  a.B = B; a.H = H; a.q0 = q0; a.out_codes = out_codes; a.out_logits = out_logits; a.forced = forced_codes;
  if (samp) { a.temperature = samp->temperature; a.top_k = samp->top_k; a.gumbel = samp->gumbel; }
  return dispatch(h, a, static_cast<cudaStream_t>(s));
}

qp_status qp_predict_frames(qp_handle* h, int B, const float* H, const int32_t* q0, int32_t* out_codes,
                            float* out_logits, qp_stream s) {
  return qp_predict_frames_ex(h, B, H, q0, out_codes, out_logits, nullptr, nullptr, s);
}

qp_status qp_predict_frames_host(qp_handle* h, int B, const float* H_host, const int32_t* q0_host,
                                 int32_t* codes_host, const qp_sampling* samp, qp_stream sv) {
  qp_status st = check_run(h, B, H_host, q0_host, codes_host, samp);
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
  st = dispatch(h, a, s);
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
  qp_status st = check_run(h, B, H, q0, out_codes, nullptr);
  if (st != QP_OK) return st;
  DeviceGuard dg(h->device);
  if (!dg.ok) return QP_ERR_CUDA;
  qp::RunArgs a;
  a.B = B; a.H = H; a.q0 = q0; a.out_codes = out_codes; a.out_logits = out_logits;
  return qp::run_frames_static(h, a, static_cast<cudaStream_t>(s));
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

int qp_launches_per_call(qp_handle* h, int B, int sampling) {
  if (!h || B < 1 || B > h->max_batch) return -1;
  static const char* eng = std::getenv("QP_ENGINE");
  if (eng && std::strcmp(eng, "layers") == 0) return qp::launches_per_call(h, B, sampling != 0);
  return 1;   // one persistent kernel per call
}

void qp_destroy(qp_handle* h) {
  if (!h) return;
  {
    DeviceGuard dg(h->device);
    cudaDeviceSynchronize();
    if (h->warena) cudaFree(h->warena);
    if (h->sarena) cudaFree(h->sarena);
  }
  delete h;
}

}  // extern "C"
