// Checkpoint I/O of a P-EAGLE draft in the layout vLLM's parallel-drafting
// loader reads ("feat(speculative): add P-EAGLE parallel-drafting training
// for EAGLE-3 drafts - #2376", Checkpoint contract): a standard EAGLE-3
// draft checkpoint -- config.json plus model.safetensors -- with the learnable
// placeholder saved under the key "mask_hidden" ([1, num_aux * target_hidden])
// and "parallel_drafting": true, "ptd_token_id" in config.json.
//
// Tensor names (the EAGLE-3 Llama draft layout; the layer index replaces l):
//   embed_tokens.weight [Vt, H]      fc.weight [H, A*Ht]   fc_norm.weight [H]
//   mask_hidden [1, A*Ht]            norm.weight [H]       lm_head.weight [Vd, H]
//   layers.l.input_layernorm.weight [H]   layers.0.hidden_norm.weight [H]
//   layers.l.self_attn.{q,k,v,o}_proj.weight   layers.l.post_attention_layernorm.weight
//   layers.l.mlp.{gate,up,down}_proj.weight
//   d2t int64 [Vd]: target id - draft id (EAGLE-3's offset form)
//   t2d bool [Vt]: target id is in the draft vocab
// The library keeps q/k/v as one [(nq+2nkv)*hd, in] matrix and gate/up as one
// [2I, H] matrix; their row blocks are the separate tensors above.
//
// safetensors: an 8-byte little-endian header length, a JSON header mapping
// each name to {dtype, shape, data_offsets}, then the raw little-endian data.
// Host code only; device weights move with cudaMemcpyAsync.
#include <ctype.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <map>
#include <memory>
#include <string>
#include <vector>

#include "common.cuh"

using namespace pe;

namespace {

// ------------------------------------------------------------------ JSON
struct Json {
  enum Kind { NUL, BOOL, NUM, STR, ARR, OBJ } kind = NUL;
  bool b = false;
  double num = 0;
  std::string str;
  std::vector<Json> arr;
  std::map<std::string, Json> obj;
  const Json* get(const std::string& k) const {
    auto it = obj.find(k);
    return (kind == OBJ && it != obj.end()) ? &it->second : nullptr;
  }
};

struct JsonParser {
  const char* p;
  const char* e;
  bool ok = true;
  void ws() {
    while (p < e && (*p == ' ' || *p == '\n' || *p == '\r' || *p == '\t')) ++p;
  }
  bool lit(const char* s) {
    const size_t n = strlen(s);
    if ((size_t)(e - p) >= n && !strncmp(p, s, n)) {
      p += n;
      return true;
    }
    return false;
  }
  std::string string() {
    std::string out;
    if (p >= e || *p != '"') {
      ok = false;
      return out;
    }
    ++p;
    while (p < e && *p != '"') {
      if (*p == '\\' && p + 1 < e) {
        ++p;
        switch (*p) {
          case 'n': out += '\n'; break;
          case 't': out += '\t'; break;
          case 'r': out += '\r'; break;
          case 'b': out += '\b'; break;
          case 'f': out += '\f'; break;
          case 'u': {   // \uXXXX: ASCII range kept, the rest replaced
            unsigned v = 0;
            for (int i = 1; i <= 4 && p + i < e; ++i) {
              const char c = p[i];
              v = v * 16 + (c >= '0' && c <= '9' ? c - '0' : (c | 32) - 'a' + 10);
            }
            out += v < 128 ? (char)v : '?';
            p += 4;
            break;
          }
          default: out += *p;
        }
        ++p;
      } else {
        out += *p++;
      }
    }
    if (p >= e) ok = false;
    ++p;
    return out;
  }
  Json value(int depth = 0) {
    Json v;
    ws();
    if (p >= e || depth > 64) {
      ok = false;
      return v;
    }
    if (*p == '{') {
      ++p;
      v.kind = Json::OBJ;
      ws();
      if (p < e && *p == '}') {
        ++p;
        return v;
      }
      while (ok) {
        ws();
        std::string k = string();
        ws();
        if (p >= e || *p != ':') {
          ok = false;
          break;
        }
        ++p;
        v.obj[k] = value(depth + 1);
        ws();
        if (p < e && *p == ',') {
          ++p;
          continue;
        }
        if (p < e && *p == '}') {
          ++p;
          break;
        }
        ok = false;
      }
    } else if (*p == '[') {
      ++p;
      v.kind = Json::ARR;
      ws();
      if (p < e && *p == ']') {
        ++p;
        return v;
      }
      while (ok) {
        v.arr.push_back(value(depth + 1));
        ws();
        if (p < e && *p == ',') {
          ++p;
          continue;
        }
        if (p < e && *p == ']') {
          ++p;
          break;
        }
        ok = false;
      }
    } else if (*p == '"') {
      v.kind = Json::STR;
      v.str = string();
    } else if (lit("true")) {
      v.kind = Json::BOOL;
      v.b = true;
    } else if (lit("false")) {
      v.kind = Json::BOOL;
    } else if (lit("null")) {
      v.kind = Json::NUL;
    } else {
      char* end = nullptr;
      std::string tok;
      while (p < e && (isdigit((unsigned char)*p) || *p == '-' || *p == '+' || *p == '.' || *p == 'e' || *p == 'E'))
        tok += *p++;
      v.num = strtod(tok.c_str(), &end);
      v.kind = Json::NUM;
      if (tok.empty() || *end) ok = false;
    }
    return v;
  }
};

bool parse_json(const std::string& text, Json* out) {
  JsonParser ps{text.data(), text.data() + text.size()};
  *out = ps.value();
  ps.ws();
  return ps.ok && ps.p == ps.e;
}

std::string json_escape(const std::string& s) {
  std::string o = "\"";
  for (char c : s) {
    if (c == '"' || c == '\\') o += '\\';
    o += c;
  }
  return o + "\"";
}

// ------------------------------------------------------------- file I/O
bool read_file(const std::string& path, std::string* out) {
  FILE* f = fopen(path.c_str(), "rb");
  if (!f) return false;
  std::string s;
  char buf[1 << 16];
  size_t n;
  while ((n = fread(buf, 1, sizeof buf, f)) > 0) s.append(buf, n);
  const bool ok = !ferror(f);
  fclose(f);
  *out = std::move(s);
  return ok;
}

// ------------------------------------------------------------- tensors
struct TensorRef {
  std::string name;
  std::string dtype;            // safetensors dtype: BF16, F32, I64, BOOL
  std::vector<int64_t> shape;
  const void* src = nullptr;    // library-layout data (device or host)
  size_t src_offset = 0;        // bytes into src
  size_t bytes = 0;
};

const char* st_dtype(int dt) { return dt == PEAGLE_BF16 ? "BF16" : "F32"; }
size_t st_esize(const std::string& d) {
  if (d == "BF16" || d == "F16") return 2;
  if (d == "F32" || d == "I32") return 4;
  if (d == "I64" || d == "F64") return 8;
  if (d == "BOOL" || d == "U8" || d == "I8") return 1;
  return 0;
}

// Every tensor of a checkpoint in file order, pointing into the library's
// weight buffers (d2t / t2d are built separately).
std::vector<TensorRef> tensor_list(const peagle_config& c, const peagle_weights& w) {
  const int H = c.hidden, A = c.num_aux, Ht = c.target_hidden, I = c.intermediate;
  const int nq = c.num_q_heads, nkv = c.num_kv_heads, hd = c.head_dim;
  const size_t es = c.dtype == PEAGLE_BF16 ? 2 : 4;
  const std::string dt = st_dtype(c.dtype);
  std::vector<TensorRef> v;
  auto add = [&](const std::string& name, std::vector<int64_t> shape, const void* src, size_t off_rows = 0,
                 int64_t row_elems = 0) {
    TensorRef t;
    t.name = name;
    t.dtype = dt;
    t.shape = shape;
    size_t n = 1;
    for (int64_t s : shape) n *= (size_t)s;
    t.bytes = n * es;
    t.src = src;
    t.src_offset = off_rows * (size_t)row_elems * es;
    v.push_back(t);
  };
  add("embed_tokens.weight", {c.target_vocab, H}, w.embed);
  add("fc.weight", {H, (int64_t)A * Ht}, w.fc_w);
  add("fc_norm.weight", {H}, w.fc_norm_w);
  add("mask_hidden", {1, (int64_t)A * Ht}, w.mask_hidden);
  for (int l = 0; l < c.num_layers; ++l) {
    const peagle_layer_weights& L = w.layers[l];
    const std::string p = "layers." + std::to_string(l) + ".";
    const int in = l == 0 ? 2 * H : H;
    add(p + "input_layernorm.weight", {H}, L.in_norm_w);
    if (l == 0) add(p + "hidden_norm.weight", {H}, L.hidden_norm_w);
    add(p + "self_attn.q_proj.weight", {(int64_t)nq * hd, in}, L.qkv_w, 0, in);
    add(p + "self_attn.k_proj.weight", {(int64_t)nkv * hd, in}, L.qkv_w, (size_t)nq * hd, in);
    add(p + "self_attn.v_proj.weight", {(int64_t)nkv * hd, in}, L.qkv_w, (size_t)(nq + nkv) * hd, in);
    add(p + "self_attn.o_proj.weight", {H, (int64_t)nq * hd}, L.o_w);
    add(p + "post_attention_layernorm.weight", {H}, L.post_norm_w);
    add(p + "mlp.gate_proj.weight", {I, H}, L.gate_up_w, 0, H);
    add(p + "mlp.up_proj.weight", {I, H}, L.gate_up_w, (size_t)I, H);
    add(p + "mlp.down_proj.weight", {H, I}, L.down_w);
  }
  add("norm.weight", {H}, w.final_norm_w);
  add("lm_head.weight", {c.draft_vocab, H}, w.lm_head_w);
  return v;
}

#define CK_FAIL(code, ...) \
  do {                     \
    set_error(__VA_ARGS__); \
    return code;           \
  } while (0)

peagle_status copy_out(void* dst, const void* src, size_t bytes, int memory, cudaStream_t s) {
  if (memory == PEAGLE_MEM_HOST) {
    memcpy(dst, src, bytes);
    return PEAGLE_OK;
  }
  cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) CK_FAIL(PEAGLE_ERR_CUDA, "checkpoint: device-to-host copy: %s", cudaGetErrorString(e));
  return PEAGLE_OK;
}

peagle_status copy_in(void* dst, const void* src, size_t bytes, int memory, cudaStream_t s) {
  if (memory == PEAGLE_MEM_HOST) {
    memcpy(dst, src, bytes);
    return PEAGLE_OK;
  }
  cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) CK_FAIL(PEAGLE_ERR_CUDA, "checkpoint: host-to-device copy: %s", cudaGetErrorString(e));
  return PEAGLE_OK;
}

peagle_status check_config(const peagle_config* c) {
  if (!c) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: config is NULL");
  if (c->dtype != PEAGLE_F32 && c->dtype != PEAGLE_BF16) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: dtype %d", c->dtype);
  if (c->hidden <= 0 || c->target_hidden <= 0 || c->num_aux <= 0 || c->num_layers <= 0 || c->num_q_heads <= 0 ||
      c->num_kv_heads <= 0 || c->head_dim <= 0 || c->intermediate <= 0 || c->target_vocab <= 0 || c->draft_vocab <= 0)
    CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: config sizes must be positive");
  if (c->draft_vocab > c->target_vocab) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: draft vocab larger than target vocab");
  if (c->ptd_token_id < 0 || c->ptd_token_id >= c->target_vocab)
    CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: ptd_token_id %d outside [0, %d)", c->ptd_token_id, c->target_vocab);
  return PEAGLE_OK;
}

std::string path_join(const char* dir, const char* name) {
  std::string p(dir);
  if (!p.empty() && p.back() != '/') p += '/';
  return p + name;
}

struct StEntry {
  std::string dtype;
  std::vector<int64_t> shape;
  size_t begin = 0, end = 0;
};

// Parses a safetensors file's header; *data_start = offset of the data.
peagle_status read_st_header(const std::string& file, std::map<std::string, StEntry>* out, size_t* data_start) {
  if (file.size() < 8) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: model.safetensors is too short");
  uint64_t n = 0;
  for (int i = 7; i >= 0; --i) n = (n << 8) | (unsigned char)file[i];
  if (n > file.size() - 8) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: safetensors header length %llu", (unsigned long long)n);
  Json h;
  if (!parse_json(file.substr(8, n), &h) || h.kind != Json::OBJ)
    CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: safetensors header is not a JSON object");
  *data_start = 8 + n;
  const size_t data_len = file.size() - *data_start;
  for (auto& kv : h.obj) {
    if (kv.first == "__metadata__") continue;
    const Json& t = kv.second;
    const Json *d = t.get("dtype"), *s = t.get("shape"), *o = t.get("data_offsets");
    if (!d || d->kind != Json::STR || !s || s->kind != Json::ARR || !o || o->kind != Json::ARR || o->arr.size() != 2)
      CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: malformed entry '%s'", kv.first.c_str());
    StEntry e;
    e.dtype = d->str;
    size_t count = 1;
    for (const Json& x : s->arr) {
      if (x.kind != Json::NUM || x.num < 0) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: bad shape of '%s'", kv.first.c_str());
      e.shape.push_back((int64_t)x.num);
      count *= (size_t)x.num;
    }
    e.begin = (size_t)o->arr[0].num;
    e.end = (size_t)o->arr[1].num;
    if (e.end < e.begin || e.end > data_len || st_esize(e.dtype) == 0 || (e.end - e.begin) != count * st_esize(e.dtype))
      CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint: entry '%s' has inconsistent dtype/shape/offsets", kv.first.c_str());
    (*out)[kv.first] = e;
  }
  return PEAGLE_OK;
}

float bf16_to_f32(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}
uint16_t f32_to_bf16(float f) {   // round to nearest even; NaN stays NaN
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

}  // namespace

extern "C" {

peagle_status peagle_checkpoint_save(const char* dir, const peagle_config* cfg, const peagle_weights* w,
                                     int32_t memory, void* stream) {
  peagle_status st = check_config(cfg);
  if (st) return st;
  if (!dir || !w || !w->layers) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_save: NULL argument");
  if (memory != PEAGLE_MEM_DEVICE && memory != PEAGLE_MEM_HOST) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_save: memory %d", memory);
  const peagle_config& c = *cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::vector<TensorRef> ts = tensor_list(c, *w);
  for (const TensorRef& t : ts)
    if (!t.src) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_save: weight for '%s' is NULL", t.name.c_str());
  // header and data offsets
  const int Vd = c.draft_vocab, Vt = c.target_vocab;
  std::string hdr = "{\"__metadata__\":{\"format\":\"pt\"}";
  size_t off = 0;
  auto entry = [&](const std::string& name, const std::string& dt, const std::vector<int64_t>& shape, size_t bytes) {
    hdr += "," + json_escape(name) + ":{\"dtype\":\"" + dt + "\",\"shape\":[";
    for (size_t i = 0; i < shape.size(); ++i) hdr += (i ? "," : "") + std::to_string(shape[i]);
    hdr += "],\"data_offsets\":[" + std::to_string(off) + "," + std::to_string(off + bytes) + "]}";
    off += bytes;
  };
  for (const TensorRef& t : ts) entry(t.name, t.dtype, t.shape, t.bytes);
  entry("d2t", "I64", {Vd}, (size_t)Vd * 8);
  entry("t2d", "BOOL", {Vt}, (size_t)Vt);
  hdr += "}";
  while ((hdr.size() + 8) % 8) hdr += ' ';
  // the vocab maps in EAGLE-3's form
  std::vector<int32_t> d2t(Vd), t2d(Vt);
  if (w->d2t) {
    st = copy_out(d2t.data(), w->d2t, (size_t)Vd * 4, memory, s);
    if (st) return st;
  }
  if (w->t2d) {
    st = copy_out(t2d.data(), w->t2d, (size_t)Vt * 4, memory, s);
    if (st) return st;
  }
  // data: one host staging buffer per tensor, written in order
  const std::string path = path_join(dir, "model.safetensors");
  std::unique_ptr<FILE, int (*)(FILE*)> f(fopen(path.c_str(), "wb"), fclose);
  if (!f) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_save: cannot write %s", path.c_str());
  unsigned char len8[8];
  for (int i = 0; i < 8; ++i) len8[i] = (unsigned char)((uint64_t)hdr.size() >> (8 * i));
  bool ok = fwrite(len8, 1, 8, f.get()) == 8 && fwrite(hdr.data(), 1, hdr.size(), f.get()) == hdr.size();
  std::vector<unsigned char> buf;
  for (const TensorRef& t : ts) {
    if (!ok) break;
    buf.resize(t.bytes);
    st = copy_out(buf.data(), static_cast<const char*>(t.src) + t.src_offset, t.bytes, memory, s);
    if (st) return st;
    if (memory == PEAGLE_MEM_DEVICE && cudaStreamSynchronize(s) != cudaSuccess)
      CK_FAIL(PEAGLE_ERR_CUDA, "checkpoint_save: stream synchronize failed");
    ok = fwrite(buf.data(), 1, t.bytes, f.get()) == t.bytes;
  }
  if (memory == PEAGLE_MEM_DEVICE && cudaStreamSynchronize(s) != cudaSuccess)
    CK_FAIL(PEAGLE_ERR_CUDA, "checkpoint_save: stream synchronize failed");
  std::vector<int64_t> off64(Vd);
  for (int j = 0; j < Vd; ++j) off64[j] = (int64_t)(w->d2t ? d2t[j] : j) - j;
  std::vector<unsigned char> mask(Vt);
  for (int t = 0; t < Vt; ++t) mask[t] = w->t2d ? (t2d[t] >= 0) : (t < Vd);
  ok = ok && fwrite(off64.data(), 8, Vd, f.get()) == (size_t)Vd && fwrite(mask.data(), 1, Vt, f.get()) == (size_t)Vt;
  if (!ok) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_save: write to %s failed", path.c_str());
  // config.json
  char num[64];
  std::string js = "{\n";
  auto kv = [&](const char* k, const std::string& v, bool last = false) {
    js += std::string("  \"") + k + "\": " + v + (last ? "\n" : ",\n");
  };
  auto dbl = [&](double x) {
    snprintf(num, sizeof num, "%.17g", x);
    return std::string(num);
  };
  kv("architectures", "[\"LlamaForCausalLMEagle3\"]");
  kv("model_type", "\"llama\"");
  kv("hidden_size", std::to_string(c.hidden));
  kv("intermediate_size", std::to_string(c.intermediate));
  kv("num_attention_heads", std::to_string(c.num_q_heads));
  kv("num_key_value_heads", std::to_string(c.num_kv_heads));
  kv("head_dim", std::to_string(c.head_dim));
  kv("num_hidden_layers", std::to_string(c.num_layers));
  kv("rms_norm_eps", dbl(c.rms_eps));
  kv("rope_theta", dbl(c.rope_theta));
  kv("max_position_embeddings", std::to_string(c.max_position));
  kv("vocab_size", std::to_string(c.target_vocab));
  kv("draft_vocab_size", std::to_string(c.draft_vocab));
  kv("target_hidden_size", std::to_string(c.target_hidden));
  kv("num_aux_hidden_states", std::to_string(c.num_aux));
  kv("norm_before_residual", c.norm_before_residual ? "true" : "false");
  kv("tie_word_embeddings", "false");
  kv("torch_dtype", c.dtype == PEAGLE_BF16 ? "\"bfloat16\"" : "\"float32\"");
  kv("parallel_drafting", "true");
  kv("ptd_token_id", std::to_string(c.ptd_token_id), true);
  js += "}\n";
  const std::string cpath = path_join(dir, "config.json");
  std::unique_ptr<FILE, int (*)(FILE*)> cf(fopen(cpath.c_str(), "wb"), fclose);
  if (!cf || fwrite(js.data(), 1, js.size(), cf.get()) != js.size())
    CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_save: cannot write %s", cpath.c_str());
  return PEAGLE_OK;
}

peagle_status peagle_checkpoint_load_config(const char* dir, peagle_config* out) {
  if (!dir || !out) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load_config: NULL argument");
  std::string text;
  const std::string cpath = path_join(dir, "config.json");
  if (!read_file(cpath, &text)) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load_config: cannot read %s", cpath.c_str());
  Json j;
  if (!parse_json(text, &j) || j.kind != Json::OBJ) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load_config: %s is not a JSON object", cpath.c_str());
  const Json* pd = j.get("parallel_drafting");
  if (!pd || pd->kind != Json::BOOL || !pd->b)
    CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load_config: config.json does not set parallel_drafting: true (not a P-EAGLE draft)");
  const Json* ptd = j.get("ptd_token_id");
  if (!ptd || ptd->kind != Json::NUM) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load_config: config.json has no ptd_token_id");
  auto need = [&](const char* k, double* v) -> bool {
    const Json* x = j.get(k);
    if (!x || x->kind != Json::NUM) return false;
    *v = x->num;
    return true;
  };
  double H, I, nq, nkv, L, Vt, eps, theta;
  if (!need("hidden_size", &H) || !need("intermediate_size", &I) || !need("num_attention_heads", &nq) ||
      !need("num_hidden_layers", &L) || !need("vocab_size", &Vt) || !need("rms_norm_eps", &eps))
    CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load_config: config.json misses a required size");
  if (!need("num_key_value_heads", &nkv)) nkv = nq;
  if (!need("rope_theta", &theta)) theta = 10000.0;
  double hd = 0, Vd = Vt, Ht = H, A = 0, maxpos = 0;
  if (!need("head_dim", &hd)) hd = H / nq;
  need("draft_vocab_size", &Vd);
  need("target_hidden_size", &Ht);
  need("max_position_embeddings", &maxpos);
  if (!need("num_aux_hidden_states", &A)) {
    const Json* ids = j.get("eagle_aux_hidden_state_layer_ids");
    if (ids && ids->kind == Json::ARR) A = (double)ids->arr.size();
  }
  if (A <= 0) {   // from the fc weight's width in the tensor header
    std::string file;
    std::map<std::string, StEntry> ents;
    size_t ds = 0;
    if (read_file(path_join(dir, "model.safetensors"), &file) && read_st_header(file, &ents, &ds) == PEAGLE_OK) {
      auto it = ents.find("fc.weight");
      if (it != ents.end() && it->second.shape.size() == 2 && Ht > 0) A = (double)it->second.shape[1] / Ht;
    }
  }
  if (A <= 0) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load_config: number of aux hidden states unknown");
  peagle_config c{};
  c.hidden = (int32_t)H;
  c.target_hidden = (int32_t)Ht;
  c.num_aux = (int32_t)A;
  c.num_layers = (int32_t)L;
  c.num_q_heads = (int32_t)nq;
  c.num_kv_heads = (int32_t)nkv;
  c.head_dim = (int32_t)hd;
  c.intermediate = (int32_t)I;
  c.target_vocab = (int32_t)Vt;
  c.draft_vocab = (int32_t)Vd;
  c.ptd_token_id = (int32_t)ptd->num;
  const Json* nbr = j.get("norm_before_residual");
  c.norm_before_residual = (nbr && nbr->kind == Json::BOOL) ? (nbr->b ? 1 : 0) : 1;
  c.max_position = (int32_t)(maxpos > 0 ? maxpos : 16384);
  const Json* td = j.get("torch_dtype");
  c.dtype = (td && td->kind == Json::STR && td->str == "float32") ? PEAGLE_F32 : PEAGLE_BF16;
  c.rope_theta = theta;
  c.rms_eps = eps;
  peagle_status st = check_config(&c);
  if (st) return st;
  *out = c;
  return PEAGLE_OK;
}

peagle_status peagle_checkpoint_load(const char* dir, const peagle_config* cfg, const peagle_weights* w,
                                     int32_t memory, void* stream) {
  peagle_status st = check_config(cfg);
  if (st) return st;
  if (!dir || !w || !w->layers) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: NULL argument");
  if (memory != PEAGLE_MEM_DEVICE && memory != PEAGLE_MEM_HOST) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: memory %d", memory);
  const peagle_config& c = *cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::string file;
  const std::string path = path_join(dir, "model.safetensors");
  if (!read_file(path, &file)) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: cannot read %s", path.c_str());
  std::map<std::string, StEntry> ents;
  size_t data0 = 0;
  st = read_st_header(file, &ents, &data0);
  if (st) return st;
  const char* data = file.data() + data0;
  std::vector<TensorRef> ts = tensor_list(c, *w);
  // every tensor is checked before any buffer is written
  for (const TensorRef& t : ts) {
    if (!t.src) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: destination for '%s' is NULL", t.name.c_str());
    auto it = ents.find(t.name);
    if (it == ents.end()) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: tensor '%s' is missing", t.name.c_str());
    const StEntry& e = it->second;
    // a [1, n] placeholder may also be stored as [n]
    const bool shape_ok =
        e.shape == t.shape || (t.name == "mask_hidden" && e.shape.size() == 1 && e.shape[0] == t.shape[1]);
    if (!shape_ok) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: '%s' has the wrong shape", t.name.c_str());
    if (e.dtype != t.dtype && !(e.dtype == "F32" || e.dtype == "BF16"))
      CK_FAIL(PEAGLE_ERR_UNSUPPORTED, "checkpoint_load: '%s' is %s, the model is %s", t.name.c_str(), e.dtype.c_str(),
              t.dtype.c_str());
  }
  // vocab maps: d2t offsets -> target ids; t2d = inverse of d2t, checked
  // against the stored membership mask
  const int Vd = c.draft_vocab, Vt = c.target_vocab;
  std::vector<int32_t> d2t(Vd), t2d(Vt, -1);
  auto id = ents.find("d2t");
  bool identity = true;
  if (id != ents.end()) {
    const StEntry& e = id->second;
    if (e.shape != std::vector<int64_t>{Vd} || (e.dtype != "I64" && e.dtype != "I32"))
      CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: d2t must be an int64 [%d] tensor", Vd);
    for (int j = 0; j < Vd; ++j) {
      int64_t o;
      if (e.dtype == "I64") {
        memcpy(&o, data + e.begin + 8 * (size_t)j, 8);
      } else {
        int32_t o32;
        memcpy(&o32, data + e.begin + 4 * (size_t)j, 4);
        o = o32;
      }
      const int64_t t = j + o;
      if (t < 0 || t >= Vt) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: d2t[%d] maps outside the target vocab", j);
      if (t2d[t] >= 0) CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: d2t maps two draft ids to target id %lld", (long long)t);
      d2t[j] = (int32_t)t;
      t2d[t] = j;
      identity = identity && (t == j);
    }
  } else {
    for (int j = 0; j < Vd; ++j) d2t[j] = t2d[j] = j;
  }
  identity = identity && Vd == Vt;
  auto im = ents.find("t2d");
  if (im != ents.end()) {
    const StEntry& e = im->second;
    if (e.shape != std::vector<int64_t>{Vt} || e.dtype != "BOOL")
      CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: t2d must be a bool [%d] tensor", Vt);
    for (int t = 0; t < Vt; ++t)
      if ((data[e.begin + t] != 0) != (t2d[t] >= 0))
        CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: t2d disagrees with d2t at target id %d", t);
  }
  if (!w->d2t && !identity)
    CK_FAIL(PEAGLE_ERR_INVALID_ARG, "checkpoint_load: the checkpoint maps draft ids to target ids; pass d2t/t2d buffers");
  std::vector<unsigned char> conv;
  for (const TensorRef& t : ts) {
    const StEntry& e = ents.find(t.name)->second;
    const char* src = data + e.begin;
    const size_t n = t.bytes / (c.dtype == PEAGLE_BF16 ? 2 : 4);
    if (e.dtype != t.dtype) {   // F32 <-> BF16 on the host
      conv.resize(t.bytes);
      if (e.dtype == "F32" && t.dtype == "BF16") {
        for (size_t i = 0; i < n; ++i) {
          float x;
          memcpy(&x, src + 4 * i, 4);
          const uint16_t b = f32_to_bf16(x);
          memcpy(conv.data() + 2 * i, &b, 2);
        }
      } else if (e.dtype == "BF16" && t.dtype == "F32") {
        for (size_t i = 0; i < n; ++i) {
          uint16_t b;
          memcpy(&b, src + 2 * i, 2);
          const float x = bf16_to_f32(b);
          memcpy(conv.data() + 4 * i, &x, 4);
        }
      } else {
        CK_FAIL(PEAGLE_ERR_UNSUPPORTED, "checkpoint_load: '%s' is %s, the model is %s", t.name.c_str(), e.dtype.c_str(),
                t.dtype.c_str());
      }
      src = reinterpret_cast<const char*>(conv.data());
    }
    void* dst = const_cast<char*>(static_cast<const char*>(t.src)) + t.src_offset;
    st = copy_in(dst, src, t.bytes, memory, s);
    if (st) return st;
    if (memory == PEAGLE_MEM_DEVICE && !conv.empty() && cudaStreamSynchronize(s) != cudaSuccess)
      CK_FAIL(PEAGLE_ERR_CUDA, "checkpoint_load: stream synchronize failed");
    conv.clear();
  }
  if (w->d2t) {
    st = copy_in(const_cast<int32_t*>(w->d2t), d2t.data(), (size_t)Vd * 4, memory, s);
    if (st) return st;
  }
  if (w->t2d) {
    st = copy_in(const_cast<int32_t*>(w->t2d), t2d.data(), (size_t)Vt * 4, memory, s);
    if (st) return st;
  }
  if (memory == PEAGLE_MEM_DEVICE && cudaStreamSynchronize(s) != cudaSuccess)
    CK_FAIL(PEAGLE_ERR_CUDA, "checkpoint_load: stream synchronize failed");
  return PEAGLE_OK;
}

}  // extern "C"
