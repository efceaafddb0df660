// Per-shape tuning table of the plan's automatic choices (Flux summary, idea
// I4: per-environment auto-tuning of one kernel code base).  The table holds
// measured best choices (tile shape, K-splits, rasterisation group, policy) per
// chain shape, row count M and grid size; cs_chain_plan applies the entry of
// the nearest measured M to every field the desc leaves on auto.  Files are
// JSON, written by the package's tuner; this file reads them.
#include <cctype>
#include <cerrno>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "cs_tune.h"

namespace {

// ------------------------------------------------------------------ JSON
// A small reader for the table files: objects, arrays, strings (escapes kept
// as given except \" \\ \/ \b \f \n \r \t; \uXXXX becomes '?'), numbers,
// true / false / null.  Nesting is limited to 32 levels.
struct JVal {
  enum Kind { Null, Bool, Num, Str, Arr, Obj } kind = Null;
  bool b = false;
  double num = 0.0;
  std::string str;
  std::vector<JVal> arr;
  std::vector<std::pair<std::string, JVal>> obj;

  const JVal* get(const char* key) const {
    for (const auto& kv : obj)
      if (kv.first == key) return &kv.second;
    return nullptr;
  }
};

class JReader {
 public:
  JReader(const char* p, size_t n) : p_(p), b_(p), e_(p + n) {}

  bool document(JVal& v) {
    if (!value(v, 0)) return false;
    space();
    if (p_ != e_) return error("trailing characters");
    return true;
  }
  const std::string& message() const { return msg_; }

 private:
  const char* p_;
  const char* b_;
  const char* e_;
  std::string msg_;

  bool error(const char* what) {
    char buf[160];
    snprintf(buf, sizeof(buf), "%s at byte %ld", what, static_cast<long>(p_ - b_));
    msg_ = buf;
    return false;
  }
  void space() {
    while (p_ < e_ && (*p_ == ' ' || *p_ == '\t' || *p_ == '\n' || *p_ == '\r')) ++p_;
  }
  bool word(const char* w) {
    const size_t n = strlen(w);
    if (static_cast<size_t>(e_ - p_) < n || strncmp(p_, w, n) != 0) return false;
    p_ += n;
    return true;
  }
  bool string(std::string& s) {
    if (p_ >= e_ || *p_ != '"') return error("expected a string");
    ++p_;
    s.clear();
    while (p_ < e_ && *p_ != '"') {
      char c = *p_++;
      if (static_cast<unsigned char>(c) < 0x20) return error("control character in a string");
      if (c == '\\') {
        if (p_ >= e_) return error("unterminated escape");
        const char x = *p_++;
        switch (x) {
          case '"': c = '"'; break;
          case '\\': c = '\\'; break;
          case '/': c = '/'; break;
          case 'b': c = '\b'; break;
          case 'f': c = '\f'; break;
          case 'n': c = '\n'; break;
          case 'r': c = '\r'; break;
          case 't': c = '\t'; break;
          case 'u':
            for (int i = 0; i < 4; ++i, ++p_)
              if (p_ >= e_ || !isxdigit(static_cast<unsigned char>(*p_))) return error("bad \\u escape");
            c = '?';
            break;
          default: return error("bad escape");
        }
      }
      s.push_back(c);
    }
    if (p_ >= e_) return error("unterminated string");
    ++p_;
    return true;
  }
  bool number(double& d) {
    // JSON grammar: -?(0|[1-9][0-9]*)(\.[0-9]+)?([eE][+-]?[0-9]+)?
    const char* s = p_;
    if (p_ < e_ && *p_ == '-') ++p_;
    if (p_ >= e_ || !isdigit(static_cast<unsigned char>(*p_))) return error("bad number");
    if (*p_ == '0') ++p_;
    else while (p_ < e_ && isdigit(static_cast<unsigned char>(*p_))) ++p_;
    if (p_ < e_ && *p_ == '.') {
      ++p_;
      if (p_ >= e_ || !isdigit(static_cast<unsigned char>(*p_))) return error("bad fraction");
      while (p_ < e_ && isdigit(static_cast<unsigned char>(*p_))) ++p_;
    }
    if (p_ < e_ && (*p_ == 'e' || *p_ == 'E')) {
      ++p_;
      if (p_ < e_ && (*p_ == '+' || *p_ == '-')) ++p_;
      if (p_ >= e_ || !isdigit(static_cast<unsigned char>(*p_))) return error("bad exponent");
      while (p_ < e_ && isdigit(static_cast<unsigned char>(*p_))) ++p_;
    }
    // The value, read by hand (strtod follows the process's locale and would stop
    // at the '.' under one with a decimal comma): integers of up to 18 digits
    // exactly, anything else as mantissa x 10^exponent in long double.
    // Underflow reads as zero; overflow is refused.
    const char* q = s;
    const bool neg = *q == '-';
    if (neg) ++q;
    long double mant = 0.0L;
    long exp10 = 0;
    int kept = 0;  // significant digits taken into the mantissa
    for (; q < p_ && isdigit(static_cast<unsigned char>(*q)); ++q) {
      if (kept < 30) mant = mant * 10.0L + (*q - '0'), kept += (mant != 0.0L);
      else ++exp10;
    }
    if (q < p_ && *q == '.')
      for (++q; q < p_ && isdigit(static_cast<unsigned char>(*q)); ++q)
        if (kept < 30) mant = mant * 10.0L + (*q - '0'), kept += (mant != 0.0L), --exp10;
    if (q < p_ && (*q == 'e' || *q == 'E')) {
      ++q;
      const bool eneg = *q == '-';
      if (*q == '+' || *q == '-') ++q;
      long e = 0;
      for (; q < p_ && isdigit(static_cast<unsigned char>(*q)); ++q)
        if (e < 100000) e = e * 10 + (*q - '0');
      exp10 += eneg ? -e : e;
    }
    if (mant == 0.0L || exp10 < -4000) {
      d = 0.0;
    } else {
      if (exp10 > 4000) return error("number out of range");
      const long double v = mant * std::pow(10.0L, static_cast<long double>(exp10));
      if (!(v <= static_cast<long double>(std::numeric_limits<double>::max()))) return error("number out of range");
      d = static_cast<double>(v);
    }
    if (neg) d = -d;
    return true;
  }
  bool value(JVal& v, int depth) {
    if (depth > 32) return error("nested too deeply");
    space();
    if (p_ >= e_) return error("unexpected end");
    const char c = *p_;
    if (c == '{') {
      ++p_;
      v.kind = JVal::Obj;
      space();
      if (p_ < e_ && *p_ == '}') return ++p_, true;
      for (;;) {
        space();
        std::pair<std::string, JVal> kv;
        if (!string(kv.first)) return false;
        space();
        if (p_ >= e_ || *p_ != ':') return error("expected ':'");
        ++p_;
        if (!value(kv.second, depth + 1)) return false;
        v.obj.push_back(std::move(kv));
        space();
        if (p_ < e_ && *p_ == ',') { ++p_; continue; }
        if (p_ < e_ && *p_ == '}') return ++p_, true;
        return error("expected ',' or '}'");
      }
    }
    if (c == '[') {
      ++p_;
      v.kind = JVal::Arr;
      space();
      if (p_ < e_ && *p_ == ']') return ++p_, true;
      for (;;) {
        JVal x;
        if (!value(x, depth + 1)) return false;
        v.arr.push_back(std::move(x));
        space();
        if (p_ < e_ && *p_ == ',') { ++p_; continue; }
        if (p_ < e_ && *p_ == ']') return ++p_, true;
        return error("expected ',' or ']'");
      }
    }
    if (c == '"') return v.kind = JVal::Str, string(v.str);
    if (word("true")) return v.kind = JVal::Bool, v.b = true, true;
    if (word("false")) return v.kind = JVal::Bool, v.b = false, true;
    if (word("null")) return v.kind = JVal::Null, true;
    return v.kind = JVal::Num, number(v.num);
  }
};

// ------------------------------------------------------------------ table
struct TuneEntry {
  int kind = 0, dtype = 0, H = 0, F = 0, M = 0, sms = 0;
  int layout = -1;  // cs_weight_layout, -1 = any
  int policy = -1;  // cs_policy, -1 = any
  int tile_m = 0, tile_n = 0, split_k = 0, group_m = 0;
  int split_k_first = 0;           // K-splits of the first stage (0: as split_k)
  int raster = 0;                  // unit order inside a row group (0: the built-in rule)
  int sk_tiles = 0, sk_units = 0;  // Stream-K tail of the last stage (0: none)
  double us = std::numeric_limits<double>::infinity();  // measured time per chain
};

std::mutex g_mu;
std::vector<TuneEntry> g_table;

struct Names {
  const char* name;
  int value;
};
const Names kKinds[] = {{"gelu", CS_CHAIN_MLP_GELU}, {"swiglu", CS_CHAIN_MLP_SWIGLU}, {"attn", CS_CHAIN_ATTN}};
const Names kDtypes[] = {{"f16", CS_F16}, {"bf16", CS_BF16}};
const Names kLayouts[] = {{"kn", CS_WEIGHTS_KN}, {"nk", CS_WEIGHTS_NK}, {"any", -1}};
const Names kPolicies[] = {{"tile", CS_SYNC_TILE}, {"row", CS_SYNC_ROW}, {"strided", CS_SYNC_STRIDED},
                           {"stream", CS_SYNC_STREAM}, {"any", -1}};

template <size_t N>
bool name_field(const JVal& o, const char* key, const Names (&names)[N], bool required, int* out, std::string& err) {
  const JVal* v = o.get(key);
  if (!v) {
    if (required) err = std::string("missing \"") + key + "\"";
    return !required;
  }
  if (v->kind == JVal::Str)
    for (const Names& n : names)
      if (v->str == n.name) return *out = n.value, true;
  err = std::string("bad \"") + key + "\"";
  return false;
}

bool int_field(const JVal& o, const char* key, int lo, int hi, bool required, int* out, std::string& err) {
  const JVal* v = o.get(key);
  if (!v) {
    if (required) err = std::string("missing \"") + key + "\"";
    return !required;
  }
  if (v->kind != JVal::Num || v->num != std::floor(v->num) || v->num < lo || v->num > hi) {
    err = std::string("\"") + key + "\" must be an integer in [" + std::to_string(lo) + ", " + std::to_string(hi) + "]";
    return false;
  }
  *out = static_cast<int>(v->num);
  return true;
}

bool read_entry(const JVal& o, TuneEntry& e, std::string& err) {
  if (o.kind != JVal::Obj) return err = "not an object", false;
  if (!name_field(o, "kind", kKinds, true, &e.kind, err) || !name_field(o, "dtype", kDtypes, true, &e.dtype, err) ||
      !name_field(o, "layout", kLayouts, false, &e.layout, err) ||
      !name_field(o, "policy", kPolicies, false, &e.policy, err) ||
      !int_field(o, "H", 8, 1 << 20, true, &e.H, err) || !int_field(o, "F", 8, 1 << 20, true, &e.F, err) ||
      !int_field(o, "M", 1, 128 * 4095, true, &e.M, err) || !int_field(o, "sms", 1, 1 << 16, true, &e.sms, err) ||
      !int_field(o, "tile_m", 0, 512, true, &e.tile_m, err) || !int_field(o, "tile_n", 0, 256, true, &e.tile_n, err) ||
      !int_field(o, "split_k", 0, 15, true, &e.split_k, err) ||
      !int_field(o, "group_m", 0, 4095, false, &e.group_m, err) ||
      !int_field(o, "split_k_first", 0, 15, false, &e.split_k_first, err) ||
      !int_field(o, "raster", 0, 3, false, &e.raster, err) ||
      !int_field(o, "sk_tiles", 0, 65534, false, &e.sk_tiles, err) ||
      !int_field(o, "sk_units", 0, 16383, false, &e.sk_units, err))
    return false;
  if (e.tile_m != 0 && e.tile_m != 128 && e.tile_m != 256 && e.tile_m != 512) return err = "bad \"tile_m\"", false;
  if (e.tile_n != 0 && e.tile_n != 64 && e.tile_n != 128 && e.tile_n != 256) return err = "bad \"tile_n\"", false;
  if (const JVal* us = o.get("us")) {
    if (us->kind != JVal::Num || !(us->num > 0.0)) return err = "\"us\" must be a positive number", false;
    e.us = us->num;
  }
  return true;
}

}  // namespace

int cs_tune_apply(const cs_chain_desc* in, int num_sms, cs_chain_desc* out) {
  *out = *in;
  if (in->tuned < 0) return -1;
  const bool tiles_auto =
      in->tile_m == 0 && in->tile_n == 0 && in->split_k == 0 && in->split_k_first == 0 && in->group_m == 0;
  const bool policy_auto = in->policy == CS_SYNC_AUTO;
  if (!tiles_auto && !policy_auto) return -1;
  std::lock_guard<std::mutex> lock(g_mu);
  auto usable = [&](const TuneEntry& e) {
    if (e.kind != in->kind || e.dtype != in->dtype || e.H != in->H || e.F != in->F || e.sms != num_sms) return false;
    if (e.layout >= 0 && e.layout != in->weight_layout) return false;
    if (policy_auto) return e.policy != CS_SYNC_STREAM;  // the two-kernel control is never picked
    return e.policy < 0 || e.policy == in->policy;
  };
  // the nearest measured M on a log scale (ties: the smaller M) ...
  int m_best = 0;
  double d_best = 0.0;
  for (const TuneEntry& e : g_table) {
    if (!usable(e)) continue;
    const double d = std::fabs(std::log2(static_cast<double>(in->M)) - std::log2(static_cast<double>(e.M)));
    if (m_best == 0 || d < d_best || (d == d_best && e.M < m_best)) m_best = e.M, d_best = d;
  }
  if (m_best == 0) return -1;
  // ... then, among that M's entries: for an auto policy the fastest; for a
  // given policy the most specific (layout and policy named), then the fastest
  int best = -1;
  for (size_t i = 0; i < g_table.size(); ++i) {
    const TuneEntry& e = g_table[i];
    if (e.M != m_best || !usable(e)) continue;
    if (best < 0) {
      best = static_cast<int>(i);
      continue;
    }
    const TuneEntry& b = g_table[best];
    const int se = (e.layout >= 0) + (e.policy >= 0), sb = (b.layout >= 0) + (b.policy >= 0);
    const bool better = policy_auto ? e.us < b.us : (se != sb ? se > sb : e.us < b.us);
    if (better) best = static_cast<int>(i);
  }
  const TuneEntry& e = g_table[best];
  if (policy_auto) out->policy = e.policy >= 0 ? e.policy : CS_SYNC_TILE;
  if (tiles_auto) {
    out->tile_m = e.tile_m;
    out->tile_n = e.tile_n;
    out->split_k = e.split_k;
    out->split_k_first = e.split_k_first;
    out->group_m = e.group_m;
    if (in->raster == 0) out->raster = e.raster;  // the desc leaves the order on auto
    if (in->sk_tiles == 0 && in->sk_units == 0) {  // the desc leaves the Stream-K tail on auto
      out->sk_tiles = e.sk_tiles;
      out->sk_units = e.sk_units;
    }
  }
  return best;
}

extern "C" {

cs_status cs_tune_load(const char* path, int* n_entries) {
  if (n_entries) *n_entries = 0;
  if (!path) return cs_fail(CS_ERR_INVALID_ARG, "path is NULL");
  FILE* f = fopen(path, "rb");
  if (!f) return cs_fail(CS_ERR_INVALID_ARG, "cannot open %s: %s", path, strerror(errno));
  std::string text;
  char buf[65536];
  size_t n;
  while ((n = fread(buf, 1, sizeof(buf), f)) > 0) {
    text.append(buf, n);
    if (text.size() > (16u << 20)) {
      fclose(f);
      return cs_fail(CS_ERR_INVALID_ARG, "%s is larger than 16 MiB", path);
    }
  }
  const bool read_error = ferror(f) != 0;
  fclose(f);
  if (read_error) return cs_fail(CS_ERR_INVALID_ARG, "cannot read %s", path);

  JVal doc;
  JReader r(text.data(), text.size());
  if (!r.document(doc)) return cs_fail(CS_ERR_INVALID_ARG, "%s: %s", path, r.message().c_str());
  const JVal* fmt = doc.kind == JVal::Obj ? doc.get("format") : nullptr;
  const JVal* ver = doc.kind == JVal::Obj ? doc.get("version") : nullptr;
  const JVal* entries = doc.kind == JVal::Obj ? doc.get("entries") : nullptr;
  if (!fmt || fmt->kind != JVal::Str || fmt->str != "cs_chain_tuning")
    return cs_fail(CS_ERR_INVALID_ARG, "%s: \"format\" is not \"cs_chain_tuning\"", path);
  if (!ver || ver->kind != JVal::Num || ver->num != 1)
    return cs_fail(CS_ERR_INVALID_ARG, "%s: unsupported \"version\" (1 is read)", path);
  if (!entries || entries->kind != JVal::Arr) return cs_fail(CS_ERR_INVALID_ARG, "%s: no \"entries\" array", path);
  std::vector<TuneEntry> table;
  table.reserve(entries->arr.size());
  for (size_t i = 0; i < entries->arr.size(); ++i) {
    TuneEntry e;
    std::string err;
    if (!read_entry(entries->arr[i], e, err))
      return cs_fail(CS_ERR_INVALID_ARG, "%s: entry %zu: %s", path, i, err.c_str());
    table.push_back(e);
  }
  std::lock_guard<std::mutex> lock(g_mu);
  g_table.swap(table);
  if (n_entries) *n_entries = static_cast<int>(g_table.size());
  return CS_OK;
}

cs_status cs_tune_clear(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_table.clear();
  return CS_OK;
}

int cs_tune_size(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  return static_cast<int>(g_table.size());
}

}  // extern "C"
