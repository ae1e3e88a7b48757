// GGUF reading for the predictor's weights: include/qp_gguf.h.
//
// Host code only.  The parser reads the header, the metadata key/values
// (keeping the numeric ones, by key) and the tensor table with plain stdio;
// tensor data is read only when qp_gguf_load_weights needs it.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <unordered_map>
#include <vector>

#include <cuda_runtime.h>

#include "qp_internal.h"
#include "../../include/qp_gguf.h"

namespace {

constexpr uint32_t kGgufMagic = 0x46554747u;   // the bytes "GGUF", little-endian
// GGML tensor types read here
constexpr uint32_t kGgmlF32 = 0, kGgmlF16 = 1, kGgmlQ8_0 = 8, kGgmlBF16 = 30;
// metadata value types
enum : uint32_t {
  kU8 = 0, kI8, kU16, kI16, kU32, kI32, kF32, kBool, kString, kArray, kU64, kI64, kF64
};

struct Tensor {
  std::string name;
  std::vector<uint64_t> dims;   // GGML order: dims[0] innermost
  uint32_t type = 0;
  uint64_t offset = 0;          // from the start of the data section
};

int scalar_size(uint32_t t) {
  switch (t) {
    case kU8: case kI8: case kBool: return 1;
    case kU16: case kI16: return 2;
    case kU32: case kI32: case kF32: return 4;
    case kU64: case kI64: case kF64: return 8;
    default: return 0;
  }
}

// Bytes of a tensor's data, or 0 for a type not read here or a size that
// does not fit in 64 bits (dimensions come from the file).
uint64_t tensor_bytes(const Tensor& t) {
  if (t.dims.empty()) return 0;
  constexpr uint64_t kMax = ~uint64_t(0);
  uint64_t n = 1;
  for (uint64_t d : t.dims) {
    if (d != 0 && n > kMax / d) return 0;
    n *= d;
  }
  switch (t.type) {
    case kGgmlF32: return n > kMax / 4 ? 0 : n * 4;
    case kGgmlF16: case kGgmlBF16: return n > kMax / 2 ? 0 : n * 2;
    case kGgmlQ8_0: return t.dims[0] % 32 || n / 32 > kMax / 34 ? 0 : n / 32 * 34;
    default: return 0;
  }
}

int dtype_of(uint32_t ggml) {
  switch (ggml) {
    case kGgmlF32: return QP_F32;
    case kGgmlF16: return QP_F16;
    case kGgmlBF16: return QP_BF16;
    case kGgmlQ8_0: return QP_Q8_0;
    default: return -1;
  }
}

// Sequential little-endian reads with a sticky failure flag.
struct Reader {
  FILE* f = nullptr;
  bool ok = true;
  bool raw(void* dst, size_t n) {
    if (ok && n && std::fread(dst, 1, n, f) != n) ok = false;
    return ok;
  }
  uint32_t u32() { uint32_t v = 0; raw(&v, 4); return v; }
  uint64_t u64() { uint64_t v = 0; raw(&v, 8); return v; }
  std::string str() {
    const uint64_t n = u64();
    if (!ok || n > (uint64_t(1) << 20)) { ok = false; return std::string(); }   // keys and names are short
    std::string s(size_t(n), '\0');
    raw(&s[0], size_t(n));
    return s;
  }
  void skip(uint64_t n) {
    if (ok && n && fseeko(f, off_t(n), SEEK_CUR) != 0) ok = false;
  }
  // skip one value of type t (arrays included); numbers are returned in *num
  void value(uint32_t t, double* num, int depth = 0) {
    if (t == kString) {
      const uint64_t n = u64();
      skip(n);
    } else if (t == kArray) {
      const uint32_t et = u32();
      const uint64_t count = u64();
      if (depth > 2) { ok = false; return; }
      const int es = scalar_size(et);
      if (es) {
        skip(count * uint64_t(es));
      } else {
        for (uint64_t i = 0; ok && i < count; ++i) value(et, nullptr, depth + 1);
      }
    } else {
      const int es = scalar_size(t);
      if (!es) { ok = false; return; }
      uint8_t b[8] = {};
      raw(b, size_t(es));
      if (num && ok) {
        switch (t) {
          case kU8: *num = b[0]; break;
          case kI8: *num = int8_t(b[0]); break;
          case kBool: *num = b[0] != 0; break;
          case kU16: { uint16_t v; std::memcpy(&v, b, 2); *num = v; break; }
          case kI16: { int16_t v; std::memcpy(&v, b, 2); *num = v; break; }
          case kU32: { uint32_t v; std::memcpy(&v, b, 4); *num = v; break; }
          case kI32: { int32_t v; std::memcpy(&v, b, 4); *num = v; break; }
          case kF32: { float v; std::memcpy(&v, b, 4); *num = v; break; }
          case kU64: { uint64_t v; std::memcpy(&v, b, 8); *num = double(v); break; }
          case kI64: { int64_t v; std::memcpy(&v, b, 8); *num = double(v); break; }
          case kF64: { double v; std::memcpy(&v, b, 8); *num = v; break; }
          default: break;
        }
      }
    }
  }
};

}  // namespace

struct qp_gguf {
  std::string path;
  std::unordered_map<std::string, double> nums;   // numeric metadata by key
  std::vector<Tensor> tensors;
  std::unordered_map<std::string, int> index;     // tensor name -> position
  uint64_t data_start = 0;
};

namespace {

const Tensor* find(const qp_gguf* f, const std::string& name) {
  if (!f) return nullptr;
  auto it = f->index.find(name);
  return it == f->index.end() ? nullptr : &f->tensors[size_t(it->second)];
}

// HF-order [out, in] of a 1- or 2-dimensional tensor (in = dims[0]).
bool hf_shape(const Tensor& t, int64_t shape[2]) {
  if (t.dims.size() == 1) { shape[0] = int64_t(t.dims[0]); shape[1] = 0; return true; }
  if (t.dims.size() == 2) { shape[0] = int64_t(t.dims[1]); shape[1] = int64_t(t.dims[0]); return true; }
  return false;
}

}  // namespace

extern "C" {

qp_status qp_gguf_open(const char* path, qp_gguf** out) {
  if (!out) return QP_ERR_ARG;
  *out = nullptr;
  if (!path) return QP_ERR_ARG;
  FILE* fp = std::fopen(path, "rb");
  if (!fp) return QP_ERR_ARG;
  Reader r;
  r.f = fp;
  auto* f = new qp_gguf;
  f->path = path;
  const uint32_t magic = r.u32(), version = r.u32();
  const uint64_t n_tensors = r.u64(), n_kv = r.u64();
  bool ok = r.ok && magic == kGgufMagic && (version == 2 || version == 3) && n_tensors < (1u << 20) &&
            n_kv < (1u << 20);
  uint64_t alignment = 32;
  for (uint64_t i = 0; ok && i < n_kv; ++i) {
    const std::string key = r.str();
    const uint32_t t = r.u32();
    double num = 0.0;
    const bool scalar = scalar_size(t) != 0;
    r.value(t, scalar ? &num : nullptr);
    if (!r.ok) { ok = false; break; }
    if (scalar) f->nums[key] = num;
    if (key == "general.alignment" && scalar) alignment = uint64_t(num);
  }
  ok = ok && alignment > 0 && (alignment & (alignment - 1)) == 0;
  for (uint64_t i = 0; ok && i < n_tensors; ++i) {
    Tensor t;
    t.name = r.str();
    const uint32_t nd = r.u32();
    if (!r.ok || nd == 0 || nd > 4) { ok = false; break; }
    for (uint32_t d = 0; d < nd; ++d) t.dims.push_back(r.u64());
    t.type = r.u32();
    t.offset = r.u64();
    if (!r.ok) { ok = false; break; }
    f->index[t.name] = int(f->tensors.size());
    f->tensors.push_back(std::move(t));
  }
  if (ok) {
    const off_t here = ftello(fp);
    ok = here >= 0;
    f->data_start = (uint64_t(here) + alignment - 1) / alignment * alignment;
    // every readable tensor's data lies inside the file
    ok = ok && fseeko(fp, 0, SEEK_END) == 0;
    const off_t end = ok ? ftello(fp) : off_t(-1);
    ok = ok && end >= 0;
    // (written so that no sum can wrap around)
    const uint64_t room = ok && uint64_t(end) >= f->data_start ? uint64_t(end) - f->data_start : 0;
    ok = ok && uint64_t(end) >= f->data_start;
    for (const Tensor& t : f->tensors) {
      const uint64_t b = tensor_bytes(t);
      if (ok && b && (t.offset % alignment || t.offset > room || b > room - t.offset)) ok = false;
    }
  }
  std::fclose(fp);
  if (!ok) {
    delete f;
    return QP_ERR_ARG;
  }
  *out = f;
  return QP_OK;
}

void qp_gguf_close(qp_gguf* f) { delete f; }

int qp_gguf_tensor_count(const qp_gguf* f) { return f ? int(f->tensors.size()) : 0; }

qp_status qp_gguf_tensor_info(const qp_gguf* f, int i, const char** name, int* dtype, int64_t shape[2]) {
  if (!f || i < 0 || i >= int(f->tensors.size())) return QP_ERR_ARG;
  const Tensor& t = f->tensors[size_t(i)];
  int64_t sh[2] = {0, 0};
  if (!hf_shape(t, sh)) return QP_ERR_ARG;
  if (name) *name = t.name.c_str();
  if (dtype) *dtype = dtype_of(t.type);
  if (shape) { shape[0] = sh[0]; shape[1] = sh[1]; }
  return QP_OK;
}

}  // extern "C"

extern "C" {

qp_status qp_gguf_geometry(const qp_gguf* pf, const qp_gguf* tf, qp_geometry* g) {
  if (!pf || !g) return QP_ERR_ARG;
  qp_geometry r;
  qp_default_geometry(&r);
  const std::string pre = "qwen3-tts.code_pred.";
  auto key_int = [&](const char* k, int& dst) {
    auto it = pf->nums.find(pre + k);
    if (it != pf->nums.end()) dst = int(it->second);
  };
  auto key_float = [&](const char* k, float& dst) {
    auto it = pf->nums.find(pre + k);
    if (it != pf->nums.end()) dst = float(it->second);
  };
  key_int("embedding_length", r.hidden);
  key_int("attention.key_length", r.head_dim);
  key_int("attention.head_count", r.n_q_heads);
  key_int("attention.head_count_kv", r.n_kv_heads);
  key_int("feed_forward_length", r.ffn);
  key_int("layer_count", r.layers);
  key_int("vocab_size", r.vocab);
  key_float("attention.layer_norm_rms_epsilon", r.rms_eps);
  key_float("rope.freq_base", r.rope_theta);
  // widths and counts the keys do not give, from the tensors
  int64_t sh[2];
  const Tensor* proj = find(pf, "code_pred.small_to_mtp_projection.weight");
  const Tensor* e0 = find(pf, "code_pred.codec_embd.0.weight");
  const Tensor* q0t = find(tf ? tf : pf, "talker.codec_embd.weight");
  if (!q0t && tf) q0t = find(pf, "talker.codec_embd.weight");
  if (!proj || !e0 || !q0t) return QP_ERR_WEIGHT_MISSING;
  if (!hf_shape(*proj, sh) || sh[1] <= 0) return QP_ERR_WEIGHT_SHAPE;
  if (sh[0] != r.hidden) return QP_ERR_WEIGHT_SHAPE;
  r.talker_hidden = int(sh[1]);
  if (!hf_shape(*e0, sh) || sh[1] <= 0) return QP_ERR_WEIGHT_SHAPE;
  if (sh[0] != r.vocab) return QP_ERR_WEIGHT_SHAPE;
  r.code_embed_dim = int(sh[1]);
  if (!hf_shape(*q0t, sh) || sh[1] != r.talker_hidden) return QP_ERR_WEIGHT_SHAPE;
  r.q0_vocab = int(sh[0]);
  int n = 0;
  while (n < 64 && find(pf, "code_pred.lm_head." + std::to_string(n) + ".weight")) ++n;
  r.n_steps = n;
  *g = r;
  return QP_OK;
}

qp_status qp_gguf_load_weights(qp_handle* h, const qp_gguf* const* files, int n_files, qp_stream sv) {
  if (!h || !files || n_files <= 0) return QP_ERR_ARG;
  for (int i = 0; i < n_files; ++i)
    if (!files[i]) return QP_ERR_ARG;
  // the tensors the predictor loads: everything named code_pred.* in any
  // file, and the q0 table; each from the first file that holds it
  struct Pick { const qp_gguf* f; const Tensor* t; };
  std::vector<Pick> picks;
  std::unordered_map<std::string, bool> taken;
  for (int i = 0; i < n_files; ++i)
    for (const Tensor& t : files[i]->tensors) {
      const bool wanted = t.name.compare(0, 10, "code_pred.") == 0 || t.name == "talker.codec_embd.weight";
      if (!wanted || taken.count(t.name)) continue;
      taken[t.name] = true;
      picks.push_back({files[i], &t});
    }
  std::vector<qp_weight> w;
  std::vector<void*> dev;
  void* host = nullptr;
  size_t host_bytes = 0;
  qp_status st = QP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(sv);
  for (const Pick& pk : picks) {
    const Tensor& t = *pk.t;
    const int dt = dtype_of(t.type);
    const uint64_t bytes = tensor_bytes(t);
    int64_t sh[2];
    if (dt < 0 || !bytes) { st = QP_ERR_WEIGHT_DTYPE; break; }
    if (!hf_shape(t, sh)) { st = QP_ERR_WEIGHT_SHAPE; break; }
    if (bytes > host_bytes) {
      if (host) cudaFreeHost(host);
      host = nullptr;
      host_bytes = 0;
      if (cudaMallocHost(&host, size_t(bytes)) != cudaSuccess) { cudaGetLastError(); st = QP_ERR_OOM; break; }
      host_bytes = size_t(bytes);
    }
    FILE* fp = std::fopen(pk.f->path.c_str(), "rb");
    const bool rd = fp && fseeko(fp, off_t(pk.f->data_start + t.offset), SEEK_SET) == 0 &&
                    std::fread(host, 1, size_t(bytes), fp) == size_t(bytes);
    if (fp) std::fclose(fp);
    if (!rd) { st = QP_ERR_ARG; break; }
    void* d = nullptr;
    if (cudaMalloc(&d, size_t(bytes)) != cudaSuccess) { cudaGetLastError(); st = QP_ERR_OOM; break; }
    dev.push_back(d);
    // the pinned buffer is reused for the next tensor: this copy completes first
    if (cudaMemcpyAsync(d, host, size_t(bytes), cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
      cudaGetLastError();
      st = QP_ERR_CUDA;
      break;
    }
    w.push_back({t.name.c_str(), qp_dtype(dt), d, {sh[0], sh[1]}});
  }
  if (st == QP_OK) st = qp_load_weights(h, w.data(), int(w.size()), sv);
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    if (st == QP_OK) st = QP_ERR_CUDA;
  }
  for (void* d : dev) cudaFree(d);
  if (host) cudaFreeHost(host);
  return st;
}

}  // extern "C"
