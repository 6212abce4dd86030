// s4kv oracle: a plain, slow, single-threaded CPU model of the int4 KIVI-style
// paged KV cache and of decode attention over it.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call
// this file; only the test suite, the smoke check and the benchmark's CPU
// baseline do. It shares no code, header, table or constant with the CUDA
// library: every rule below is restated here from the method's description.
//
// Sources (web pages on the method, cited by page and section):
//  * "4.4 KV Cache 量化" (infra-guide), section 3.1: keys are grouped per channel
//    over consecutive tokens, values per token over channel groups; inside a
//    group the mapping is asymmetric, from the group minimum and maximum; b bits
//    give 2^b codes.
//  * same page, section 3.2: a full-precision residual holds new key tokens
//    until a group is full, then the group is quantized as a batch into the
//    history; the value residual is a sliding window of the newest tokens, each
//    arrival evicting (and quantizing) the oldest.
//  * same page, section 2: P = softmax(Q K^T / sqrt(d)), output P V.
//  * same page, section 1: M_KV = 2 L B T H_KV d b.
//  * "给 KV cache 减肥" (ai-reference-codex), section 3.1: compress before the
//    write, restore before the product with the next query.
//  * S4 KV product page: head_dim 128, standard attention; unsupported models
//    fail fast.
//
// Where those pages are silent the readings are:
//  * scale s = (max - min) / (2^b - 1), stored with min (fp32 each); code
//    c = clamp(round_half_even((x - min) / s), 0, 2^b - 1); s == 0 gives c = 0.
//  * min and max are canonicalised with "+ 0.0f" so a -0 never reaches the
//    metadata.
//  * dequantisation is fmaf(c, s, min): one rounding.
//  * the value channel group is Gv channels (Gv = G in the shipped configs).
//  * query head h reads KV head h / (H_q / H_kv).
//  * bits = 8 selects FP8 E4M3 pages instead of KIVI codes (same page and block
//    table machinery): each token is stored on arrival, element by element, as
//    the saturating round-to-nearest-even e4m3 of x / scale, the division
//    rounded to binary32 first; scale is one float per KV head and tensor (keys,
//    values), 1.0 unless set; the restored element is value(code) * scale.
// Build: g++ -O2 -ffp-contract=off -std=c++17 (no fast-math), so every float
// operation is one IEEE-754 binary32 operation rounded to nearest-even.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <limits>
#include <cstring>
#include <deque>
#include <vector>

namespace {

// ---- narrow -> fp32, bit-exact, written from the IEEE-754 formats -------------
float half_bits_to_float(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int expo = (h >> 10) & 0x1f;
  const int frac = h & 0x3ff;
  float v;
  if (expo == 0) {
    v = std::ldexp(static_cast<float>(frac), -24);           // subnormal / zero
  } else if (expo == 31) {
    v = frac ? std::nanf("") : INFINITY;
  } else {
    v = std::ldexp(static_cast<float>(frac | 0x400), expo - 25);  // 1.frac * 2^(e-15)
  }
  return sign ? -v : v;
}

float bf16_bits_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;   // bf16 is the top half of binary32
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

enum { ORC_F16 = 0, ORC_BF16 = 1 };

float widen(uint16_t bits, int dtype) {
  return dtype == ORC_BF16 ? bf16_bits_to_float(bits) : half_bits_to_float(bits);
}

// ---- the min/max asymmetric quantizer of one group ------------------------------
// x[i * stride], i < n. Writes codes[i * code_stride] (one code per byte).
void quantize_group(const float* x, int n, int stride, int bits, float* scale_out,
                    float* min_out, uint8_t* codes, int code_stride) {
  const int levels = (1 << bits) - 1;
  float lo = x[0], hi = x[0];
  for (int i = 1; i < n; ++i) {
    const float v = x[static_cast<long>(i) * stride];
    if (v < lo) lo = v;
    if (v > hi) hi = v;
  }
  lo = lo + 0.0f;   // -0 -> +0
  hi = hi + 0.0f;
  const float range = hi - lo;
  const float s = range / static_cast<float>(levels);
  *scale_out = s;
  *min_out = lo;
  for (int i = 0; i < n; ++i) {
    int c = 0;
    if (s != 0.0f) {
      const float t = (x[static_cast<long>(i) * stride] - lo) / s;
      c = static_cast<int>(std::nearbyint(t));   // default rounding mode: half to even
      if (c < 0) c = 0;
      if (c > levels) c = levels;
    }
    codes[static_cast<long>(i) * code_stride] = static_cast<uint8_t>(c);
  }
}

float dequant(int code, float s, float mn) {
  return std::fma(static_cast<float>(code), s, mn);
}

// ---- FP8 E4M3 pages ("4.4 KV Cache 量化", sections 4.1 and 4.2: the fp8_e4m3
// KV cache type, a scale per attention head that is 1.0 unless calibrated) -----
// Bits s eeee mmm, exponent bias 7: e = 0 gives m * 2^-9 (subnormal), otherwise
// (1 + m/8) * 2^(e-7); e = 15 with m = 7 is NaN, so the largest finite value is
// 1.75 * 2^8 = 448. There is no infinity.
float e4m3_decode(uint8_t code) {
  const int sgn = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return std::numeric_limits<float>::quiet_NaN();
  const double mag = e == 0 ? std::ldexp(static_cast<double>(m), -9)
                            : std::ldexp(1.0 + m / 8.0, e - 7);
  return static_cast<float>(sgn ? -mag : mag);
}

// Nearest E4M3 value with ties to the even mantissa; magnitudes from 448 up
// saturate to 448 (the saturating conversion); the sign of zero is kept. Codes
// 0 .. 126 increase with magnitude with no gap: in the binade [2^E, 2^(E+1)),
// E >= -6, the step is 2^(E-3) and code = a / step + 8 (E + 6); below 2^-6 the
// subnormals use the same step as E = -6.
uint8_t e4m3_encode(float y) {
  const uint8_t sgn = std::signbit(y) ? 0x80 : 0x00;
  if (std::isnan(y)) return static_cast<uint8_t>(sgn | 0x7f);
  const double a = std::fabs(static_cast<double>(y));
  if (a >= 448.0) return static_cast<uint8_t>(sgn | 0x7e);
  int ex = 0;
  std::frexp(a, &ex);                                   // a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
  const int E = a == 0.0 ? -6 : std::max(ex - 1, -6);
  const double q = std::nearbyint(std::ldexp(a, 3 - E));   // exact quotient a / 2^(E-3), half-even
  const long code = static_cast<long>(q) + 8L * (E + 6);
  return static_cast<uint8_t>(sgn | code);
}

}  // namespace

extern "C" {

typedef struct {
  int head_dim;      // d
  int num_kv_heads;  // H_kv
  int group_k;       // G: tokens per key group (per channel)
  int group_v;       // Gv: channels per value group (per token)
  int residual_v;    // R: value sliding-window length
  int page_size;     // P: tokens per physical page
  int dtype;         // 0 fp16, 1 bf16 (the raw input format)
  int bits;          // code width (4 for this cache)
} orc_cfg;

int orc_version(void) { return 1; }

float orc_widen(uint16_t bits, int dtype) { return widen(bits, dtype); }

void orc_widen_array(const uint16_t* in, long n, int dtype, float* out) {
  for (long i = 0; i < n; ++i) out[i] = widen(in[i], dtype);
}

void orc_quantize_group(const float* x, int n, int stride, int bits, float* scale,
                        float* mn, uint8_t* codes, int code_stride) {
  quantize_group(x, n, stride, bits, scale, mn, codes, code_stride);
}

float orc_dequant(int code, float s, float mn) { return dequant(code, s, mn); }

// M_KV = 2 * L * B * T * H_KV * d * b (bytes; b = bytes per element).
double orc_mkv_bytes(double L, double B, double T, double H, double d, double b) {
  return 2.0 * L * B * T * H * d * b;
}

// ---- one sequence's cache state, advanced token by token ------------------------
struct orc_seq {
  orc_cfg cfg;
  long T = 0;
  std::vector<std::vector<uint8_t>> kcode;  // [h] -> Tk * d codes
  std::vector<std::vector<float>> ks, kmn;  // [h] -> (Tk / G) * d
  std::vector<std::vector<uint8_t>> vcode;  // [h] -> Tv * d codes
  std::vector<std::vector<float>> vs, vmn;  // [h] -> Tv * (d / Gv)
  std::vector<std::deque<std::vector<uint16_t>>> kres, vres;  // [h] -> raw rows
  long Tk = 0, Tv = 0;
  // FP8 pages (bits = 8): every token is encoded on arrival, x -> e4m3(x / scale)
  std::vector<float> k8s, v8s;                   // [h] per-head scales (1.0 unless set)
};

orc_seq* orc_seq_new(const orc_cfg* c) {
  if (!c || c->head_dim <= 0 || c->num_kv_heads <= 0 || c->group_k <= 0 ||
      c->group_v <= 0 || c->head_dim % c->group_v != 0 || c->residual_v < 0 ||
      c->bits < 1 || c->bits > 8 || (c->dtype != ORC_F16 && c->dtype != ORC_BF16))
    return nullptr;
  orc_seq* s = new orc_seq;
  s->cfg = *c;
  const int H = c->num_kv_heads;
  s->kcode.resize(H); s->ks.resize(H); s->kmn.resize(H);
  s->vcode.resize(H); s->vs.resize(H); s->vmn.resize(H);
  s->kres.resize(H); s->vres.resize(H);
  s->k8s.assign(H, 1.0f);
  s->v8s.assign(H, 1.0f);
  return s;
}

// Per-head FP8 scales (bits = 8), set before the first append.
void orc_seq_set_fp8_scales(orc_seq* s, const float* kscale, const float* vscale) {
  for (int h = 0; h < s->cfg.num_kv_heads; ++h) {
    s->k8s[h] = kscale[h];
    s->v8s[h] = vscale[h];
  }
}

uint8_t orc_e4m3_encode(float y) { return e4m3_encode(y); }
float orc_e4m3_decode(uint8_t code) { return e4m3_decode(code); }

void orc_seq_free(orc_seq* s) { delete s; }

// Appends n tokens; k and v are raw rows [n][H_kv][d].
// Key path: the newest token joins the key residual; once it holds G tokens the
// whole group is quantized channel by channel and moves to the history.
// Value path: the newest token joins the window; when the window exceeds R the
// oldest token leaves it and is quantized over its channel groups.
int orc_seq_append(orc_seq* s, const uint16_t* k, const uint16_t* v, long n) {
  const orc_cfg& c = s->cfg;
  const int H = c.num_kv_heads, d = c.head_dim, G = c.group_k, Gv = c.group_v;
  if (c.bits == 8) {   // FP8 pages: no residual, one code per element, x / scale rounded once in fp32
    for (long i = 0; i < n; ++i) {
      for (int h = 0; h < H; ++h) {
        for (int ch = 0; ch < d; ++ch) {
          const float kx = widen(k[(i * H + h) * d + ch], c.dtype) / s->k8s[h];
          const float vx = widen(v[(i * H + h) * d + ch], c.dtype) / s->v8s[h];
          s->kcode[h].push_back(e4m3_encode(kx));
          s->vcode[h].push_back(e4m3_encode(vx));
        }
      }
      s->T += 1;
    }
    s->Tk = s->Tv = s->T;
    return 0;
  }
  std::vector<float> buf(static_cast<size_t>(G) * d);
  std::vector<uint8_t> codes(static_cast<size_t>(G) * d);
  std::vector<float> row(d);
  std::vector<uint8_t> rowc(d);
  for (long i = 0; i < n; ++i) {
    for (int h = 0; h < H; ++h) {
      const uint16_t* krow = k + (i * H + h) * d;
      const uint16_t* vrow = v + (i * H + h) * d;
      s->kres[h].emplace_back(krow, krow + d);
      if (static_cast<int>(s->kres[h].size()) == G) {
        for (int t = 0; t < G; ++t)
          for (int ch = 0; ch < d; ++ch) buf[t * d + ch] = widen(s->kres[h][t][ch], c.dtype);
        std::vector<float> sc(d), mn(d);
        for (int ch = 0; ch < d; ++ch)   // one group per channel, down the G tokens
          quantize_group(&buf[ch], G, d, c.bits, &sc[ch], &mn[ch], &codes[ch], d);
        s->kcode[h].insert(s->kcode[h].end(), codes.begin(), codes.end());
        s->ks[h].insert(s->ks[h].end(), sc.begin(), sc.end());
        s->kmn[h].insert(s->kmn[h].end(), mn.begin(), mn.end());
        s->kres[h].clear();
      }
      s->vres[h].emplace_back(vrow, vrow + d);
      if (static_cast<int>(s->vres[h].size()) > c.residual_v) {
        const std::vector<uint16_t> old = s->vres[h].front();
        s->vres[h].pop_front();
        for (int ch = 0; ch < d; ++ch) row[ch] = widen(old[ch], c.dtype);
        for (int g = 0; g < d / Gv; ++g) {   // one group per channel block, along one token
          float sc, mn;
          quantize_group(&row[g * Gv], Gv, 1, c.bits, &sc, &mn, &rowc[g * Gv], 1);
          s->vs[h].push_back(sc);
          s->vmn[h].push_back(mn);
        }
        s->vcode[h].insert(s->vcode[h].end(), rowc.begin(), rowc.end());
      }
    }
    s->T += 1;
    s->Tk = static_cast<long>(s->kcode[0].size()) / d;
    s->Tv = static_cast<long>(s->vcode[0].size()) / d;
  }
  return 0;
}

// counts[0..4] = T, Tk (quantized keys), Tv (quantized values), key residual
// rows, value residual rows.
void orc_seq_counts(const orc_seq* s, long* counts) {
  counts[0] = s->T;
  counts[1] = s->Tk;
  counts[2] = s->Tv;
  counts[3] = static_cast<long>(s->kres[0].size());
  counts[4] = static_cast<long>(s->vres[0].size());
}

// Logical history of head h: key codes [Tk][d], key scale/min [Tk/G][d],
// value codes [Tv][d], value scale/min [Tv][d/Gv]. Null pointers are skipped.
void orc_seq_history(const orc_seq* s, int h, uint8_t* kcode, float* ks, float* kmn,
                     uint8_t* vcode, float* vs, float* vmn) {
  if (kcode) std::memcpy(kcode, s->kcode[h].data(), s->kcode[h].size());
  if (ks) std::memcpy(ks, s->ks[h].data(), s->ks[h].size() * 4);
  if (kmn) std::memcpy(kmn, s->kmn[h].data(), s->kmn[h].size() * 4);
  if (vcode) std::memcpy(vcode, s->vcode[h].data(), s->vcode[h].size());
  if (vs) std::memcpy(vs, s->vs[h].data(), s->vs[h].size() * 4);
  if (vmn) std::memcpy(vmn, s->vmn[h].data(), s->vmn[h].size() * 4);
}

// Restored K^, V^ of head h, [T][d] fp32: the history through fmaf(code, s, min),
// the residual rows widened exactly.
void orc_seq_dequant(const orc_seq* s, int h, float* khat, float* vhat) {
  const orc_cfg& c = s->cfg;
  const int d = c.head_dim, G = c.group_k, Gv = c.group_v, ng = d / Gv;
  if (c.bits == 8) {
    for (long t = 0; t < s->T; ++t) {
      for (int ch = 0; ch < d; ++ch) {
        if (khat) khat[t * d + ch] = e4m3_decode(s->kcode[h][t * d + ch]) * s->k8s[h];
        if (vhat) vhat[t * d + ch] = e4m3_decode(s->vcode[h][t * d + ch]) * s->v8s[h];
      }
    }
    return;
  }
  for (long t = 0; t < s->T; ++t) {
    for (int ch = 0; ch < d; ++ch) {
      float kv;
      if (t < s->Tk) {
        const long g = t / G;
        kv = dequant(s->kcode[h][t * d + ch], s->ks[h][g * d + ch], s->kmn[h][g * d + ch]);
      } else {
        kv = widen(s->kres[h][t - s->Tk][ch], c.dtype);
      }
      float vv;
      if (t < s->Tv) {
        const int g = ch / Gv;
        vv = dequant(s->vcode[h][t * d + ch], s->vs[h][t * ng + g], s->vmn[h][t * ng + g]);
      } else {
        vv = widen(s->vres[h][t - s->Tv][ch], c.dtype);
      }
      if (khat) khat[t * d + ch] = kv;
      if (vhat) vhat[t * d + ch] = vv;
    }
  }
}

// Decode attention for one query row against restored K^, V^ ([T][d] fp32):
// z_t = sm_scale * sum_c q_c k_tc, p = softmax(z), o = sum_t p_t v_t.
// Everything in double; the result is rounded once to fp32. T == 0 gives zeros.
void orc_attention_row(const float* q, const float* khat, const float* vhat, long T, int d,
                       float sm_scale, float* out) {
  if (T <= 0) {
    for (int c = 0; c < d; ++c) out[c] = 0.0f;
    return;
  }
  std::vector<double> z(T);
  double m = -INFINITY;
  for (long t = 0; t < T; ++t) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += static_cast<double>(q[c]) * static_cast<double>(khat[t * d + c]);
    z[t] = static_cast<double>(sm_scale) * acc;
    if (z[t] > m) m = z[t];
  }
  double l = 0.0;
  for (long t = 0; t < T; ++t) {
    z[t] = std::exp(z[t] - m);
    l += z[t];
  }
  std::vector<double> o(d, 0.0);
  for (long t = 0; t < T; ++t)
    for (int c = 0; c < d; ++c) o[c] += z[t] * static_cast<double>(vhat[t * d + c]);
  for (int c = 0; c < d; ++c) out[c] = static_cast<float>(o[c] / l);
}

// Decode attention of g query heads that share KV head h of this sequence.
// q: raw rows [g][d] in the cache dtype. out: [g][d] fp32.
void orc_seq_attention(const orc_seq* s, int h, const uint16_t* q, int g, float sm_scale,
                       float* out) {
  const int d = s->cfg.head_dim;
  std::vector<float> khat(static_cast<size_t>(s->T) * d), vhat(static_cast<size_t>(s->T) * d);
  orc_seq_dequant(s, h, khat.data(), vhat.data());
  std::vector<float> qf(d);
  for (int j = 0; j < g; ++j) {
    for (int c = 0; c < d; ++c) qf[c] = widen(q[j * d + c], s->cfg.dtype);
    orc_attention_row(qf.data(), khat.data(), vhat.data(), s->T, d, sm_scale, out + j * d);
  }
}

// Causal attention of nq query tokens that end the sequence (the chunk of a
// chunked prefill, or the tokens a speculative step verifies), for the g query
// heads of KV head h. The chunk has been appended: the state is the canonical
// state of length T. Query i sits at position T - nq + i and attends to tokens
// 0 .. T - nq + i of that state (causal mask); each row is orc_attention_row
// over that prefix of K^, V^. q: raw rows [nq][g][d]; out: [nq][g][d] fp32.
// Returns -1 (and writes nothing) when nq > T.
int orc_seq_attention_causal(const orc_seq* s, int h, const uint16_t* q, int nq, int g, float sm_scale,
                             float* out) {
  if (nq < 1 || nq > s->T) return -1;
  const int d = s->cfg.head_dim;
  std::vector<float> khat(static_cast<size_t>(s->T) * d), vhat(static_cast<size_t>(s->T) * d);
  orc_seq_dequant(s, h, khat.data(), vhat.data());
  std::vector<float> qf(d);
  for (int i = 0; i < nq; ++i) {
    const long visible = s->T - nq + i + 1;
    for (int j = 0; j < g; ++j) {
      const long row = static_cast<long>(i) * g + j;
      for (int c = 0; c < d; ++c) qf[c] = widen(q[row * d + c], s->cfg.dtype);
      orc_attention_row(qf.data(), khat.data(), vhat.data(), visible, d, sm_scale, out + row * d);
    }
  }
  return 0;
}

// ---- physical image of the paged format ----------------------------------------
// The byte format of one (page, kv head) record, 3072 bytes, for d = 128,
// P = 16, G = 32, Gv = 32, 4-bit codes. Offsets inside the record:
//   [0, 1024)    key codes     [1024, 1536) key scale/min
//   [1536, 2560) value codes   [2560, 3072) value scale/min
// Lane L = 4*a + b (a in 0..7, b in 0..3). Page-local token tau in 0..15.
// Key codes: word (kk, L), kk in 0..7, at byte (kk/4)*512 + L*16 + (kk%4)*4.
//   It holds channels c_j = 32*b + 4*kk + j of tokens a (low nibbles) and a+8
//   (high nibbles); byte 0 <- c_0, byte 1 <- c_2, byte 2 <- c_1, byte 3 <- c_3.
// Key scale/min: the group's 32 tokens span pages 2m and 2m+1; page 2m+j holds
//   channels 64j .. 64j+63. Channel 64j + 32*u + 4*i + e (u in 0..1, i in 0..7,
//   e in 0..3): scale at byte 1024 + (2i+u)*16 + 4e, min 256 bytes later.
// Value codes: word (mt, L), mt in 0..7, at byte 1536 + (mt/4)*512 + L*16 + (mt%4)*4.
//   Low nibble = channel 16*mt + a, high nibble = channel 16*mt + a + 8;
//   byte 0 <- token 2b, byte 1 <- token 2b+8, byte 2 <- token 2b+1, byte 3 <- token 2b+9.
// Value scale/min: token tau = 2b + r + 8w (r, w in 0..1) is slot e = r + 2w of
//   lane-column b. Its group k (channels 32k .. 32k+31) scale sits at byte
//   2560 + ((2k)*4 + b)*16 + 4e and its min at 2560 + ((2k+1)*4 + b)*16 + 4e.

enum { REC = 3072, KC = 0, KM = 1024, VC = 1536, VM = 2560 };

static void put_nibble(uint8_t* rec, uint8_t* valid, long off, int high, int code) {
  uint8_t b = rec[off];
  if (high) b = static_cast<uint8_t>((b & 0x0f) | (code << 4));
  else b = static_cast<uint8_t>((b & 0xf0) | code);
  rec[off] = b;
  if (valid) valid[off] |= static_cast<uint8_t>(high ? 0xf0 : 0x0f);
}

static void put_f32(uint8_t* rec, uint8_t* valid, long off, float f) {
  std::memcpy(rec + off, &f, 4);
  if (valid) std::memset(valid + off, 0xff, 4);
}

// The 2-bit record, 2048 bytes: [0, 512) key codes, [512, 1024) key scale/min,
// [1024, 1536) value codes, [1536, 2048) value scale/min. A byte holds four 2-bit
// codes; "position p" is bits 2p .. 2p+1.
// Key codes: word (kp, L), kp in 0..3, at byte L*16 + kp*4 covers the channels
//   c_j = 32*b + 4*kk + j of kk = 2kp and 2kp+1; byte 0 <- c_0, byte 1 <- c_2,
//   byte 2 <- c_1, byte 3 <- c_3; in a byte, position 0 <- (token a, kk = 2kp),
//   1 <- (token a+8, 2kp), 2 <- (token a, 2kp+1), 3 <- (token a+8, 2kp+1).
// Key scale/min: as in the 4-bit record, 512 bytes earlier (at 512).
// Value codes: word (mp, L), mp in 0..3, at byte 1024 + L*16 + mp*4; bytes hold
//   tokens as in the 4-bit record (0 <- 2b, 1 <- 2b+8, 2 <- 2b+1, 3 <- 2b+9); in a
//   byte, position q (0..3) <- channel 32*mp + 8*q + a.
// Value scale/min: as in the 4-bit record, at 1536.
enum { REC2 = 2048, KC2 = 0, KM2 = 512, VC2 = 1024, VM2 = 1536 };

static void put_crumb(uint8_t* rec, uint8_t* valid, long off, int pos, int code) {
  const uint8_t mask = static_cast<uint8_t>(3u << (2 * pos));
  rec[off] = static_cast<uint8_t>((rec[off] & ~mask) | ((code & 3) << (2 * pos)));
  if (valid) valid[off] |= mask;
}

static int page_image_2bit(const orc_seq* s, const int32_t* bt, long num_pages, uint8_t* pages,
                           uint8_t* valid) {
  const orc_cfg& c = s->cfg;
  const int H = c.num_kv_heads, d = 128;
  auto rec_of = [&](long tok, int h, uint8_t** r, uint8_t** vm) -> int {
    const long pp = bt[tok / 16];
    if (pp < 0 || pp >= num_pages) return -2;
    *r = pages + (pp * H + h) * REC2;
    *vm = valid ? valid + (pp * H + h) * REC2 : nullptr;
    return 0;
  };
  static const int byte_of_j[4] = {0, 2, 1, 3};
  static const int byte_of_tok[2][2] = {{0, 2}, {1, 3}};  // [w][r]
  for (int h = 0; h < H; ++h) {
    for (long t = 0; t < s->Tk; ++t) {
      uint8_t *r, *vmask;
      if (rec_of(t, h, &r, &vmask)) return -2;
      const int tau = static_cast<int>(t % 16), a = tau % 8, hi = tau / 8;
      for (int ch = 0; ch < d; ++ch) {
        const int b = ch / 32, kk = (ch % 32) / 4, j = ch % 4;
        const long off = KC2 + (4 * a + b) * 16 + (kk / 2) * 4 + byte_of_j[j];
        put_crumb(r, vmask, off, 2 * (kk % 2) + hi, s->kcode[h][t * d + ch]);
      }
    }
    for (long grp = 0; grp < s->Tk / 32; ++grp) {
      for (int j = 0; j < 2; ++j) {
        uint8_t *r, *vmask;
        if (rec_of(grp * 32 + 16 * j, h, &r, &vmask)) return -2;
        for (int cl = 0; cl < 64; ++cl) {
          const int ch = 64 * j + cl, u = cl / 32, i = (cl % 32) / 4, e = cl % 4;
          const long off = KM2 + (2 * i + u) * 16 + 4 * e;
          put_f32(r, vmask, off, s->ks[h][grp * d + ch]);
          put_f32(r, vmask, off + 256, s->kmn[h][grp * d + ch]);
        }
      }
    }
    for (long t = 0; t < s->Tv; ++t) {
      uint8_t *r, *vmask;
      if (rec_of(t, h, &r, &vmask)) return -2;
      const int tau = static_cast<int>(t % 16), w = tau / 8, b = (tau % 8) / 2, rr = tau % 2;
      for (int ch = 0; ch < d; ++ch) {
        const int mp = ch / 32, q = (ch % 32) / 8, a = ch % 8;
        const long off = VC2 + (4 * a + b) * 16 + mp * 4 + byte_of_tok[w][rr];
        put_crumb(r, vmask, off, q, s->vcode[h][t * d + ch]);
      }
      const int e = rr + 2 * w;
      for (int k = 0; k < 4; ++k) {
        put_f32(r, vmask, VM2 + ((2 * k) * 4 + b) * 16 + 4 * e, s->vs[h][t * 4 + k]);
        put_f32(r, vmask, VM2 + ((2 * k + 1) * 4 + b) * 16 + 4 * e, s->vmn[h][t * 4 + k]);
      }
    }
  }
  return 0;
}

// The FP8 record (bits = 8), 4096 bytes: [0, 2048) keys, [2048, 4096) values, one
// e4m3 byte per element. Lane L = 4a + b as above; word (kp, L), kp in 0..3, is
// the 16 bytes at kp*512 + L*16 of a half.
// Keys: the word's bytes 8u .. 8u+7 hold slice kk = 2kp + u (channels c_j =
//   32b + 4kk + j): byte 8u + 4*(j/2) + 2*hi + (j%2) <- (token a + 8*hi, c_j).
// Values: the word's bytes 8u .. 8u+7 hold tile mt = 2kp + u (channels 16mt + a
//   + 8*up): token tau = 2b + r + 8w goes to byte 8u + 4w + 2*up + r.
enum { REC8 = 4096, K8 = 0, V8 = 2048 };

static int page_image_fp8(const orc_seq* s, const int32_t* bt, long num_pages, uint8_t* pages, uint8_t* valid) {
  const int H = s->cfg.num_kv_heads, d = 128;
  for (int h = 0; h < H; ++h) {
    for (long t = 0; t < s->T; ++t) {
      const long pp = bt[t / 16];
      if (pp < 0 || pp >= num_pages) return -2;
      uint8_t* r = pages + (pp * H + h) * REC8;
      uint8_t* vm = valid ? valid + (pp * H + h) * REC8 : nullptr;
      const int tau = static_cast<int>(t % 16);
      for (int ch = 0; ch < d; ++ch) {
        {   // key
          const int a = tau % 8, hi = tau / 8, b = ch / 32, kk = (ch % 32) / 4, j = ch % 4;
          const long off = K8 + (kk / 2) * 512 + (4 * a + b) * 16 + 8 * (kk % 2) + 4 * (j / 2) + 2 * hi + (j % 2);
          r[off] = s->kcode[h][t * d + ch];
          if (vm) vm[off] = 0xff;
        }
        {   // value
          const int mt = ch / 16, a = ch % 8, up = (ch % 16) / 8;
          const int b = (tau % 8) / 2, rr = tau % 2, w = tau / 8;
          const long off = V8 + (mt / 2) * 512 + (4 * a + b) * 16 + 8 * (mt % 2) + 4 * w + 2 * up + rr;
          r[off] = s->vcode[h][t * d + ch];
          if (vm) vm[off] = 0xff;
        }
      }
    }
  }
  return 0;
}

// pages: [num_pages][H][record] image (3072-byte records for 4-bit codes, 2048
// for 2-bit, 4096 for FP8); valid: same shape, bit mask of defined bits. bt: block-table row
// (logical page -> physical page). Returns 0, or -1 when the configuration is
// not one the physical format is defined for, -2 when a block-table entry is
// out of range.
int orc_seq_page_image(const orc_seq* s, const int32_t* bt, long num_pages, uint8_t* pages,
                       uint8_t* valid) {
  const orc_cfg& c = s->cfg;
  if (c.head_dim != 128 || c.page_size != 16 || c.group_k != 32 || c.group_v != 32 ||
      (c.bits != 4 && c.bits != 2 && c.bits != 8))
    return -1;
  if (c.bits == 2) return page_image_2bit(s, bt, num_pages, pages, valid);
  if (c.bits == 8) return page_image_fp8(s, bt, num_pages, pages, valid);
  const int H = c.num_kv_heads, d = 128;
  auto rec_of = [&](long tok, int h, uint8_t** r, uint8_t** vm) -> int {
    const long lp = tok / 16;
    const long pp = bt[lp];
    if (pp < 0 || pp >= num_pages) return -2;
    *r = pages + (pp * H + h) * REC;
    *vm = valid ? valid + (pp * H + h) * REC : nullptr;
    return 0;
  };
  for (int h = 0; h < H; ++h) {
    // keys
    for (long t = 0; t < s->Tk; ++t) {
      uint8_t *r, *vmask;
      if (rec_of(t, h, &r, &vmask)) return -2;
      const int tau = static_cast<int>(t % 16);
      const int a = tau % 8, high = tau / 8;
      for (int ch = 0; ch < d; ++ch) {
        const int b = ch / 32, kk = (ch % 32) / 4, j = ch % 4;
        static const int byte_of_j[4] = {0, 2, 1, 3};
        const int L = 4 * a + b;
        const long off = KC + (kk / 4) * 512 + L * 16 + (kk % 4) * 4 + byte_of_j[j];
        put_nibble(r, vmask, off, high, s->kcode[h][t * d + ch]);
      }
    }
    for (long grp = 0; grp < s->Tk / 32; ++grp) {
      for (int j = 0; j < 2; ++j) {
        uint8_t *r, *vmask;
        if (rec_of(grp * 32 + 16 * j, h, &r, &vmask)) return -2;
        for (int cl = 0; cl < 64; ++cl) {
          const int ch = 64 * j + cl;
          const int u = cl / 32, i = (cl % 32) / 4, e = cl % 4;
          const long off = KM + (2 * i + u) * 16 + 4 * e;
          put_f32(r, vmask, off, s->ks[h][grp * d + ch]);
          put_f32(r, vmask, off + 256, s->kmn[h][grp * d + ch]);
        }
      }
    }
    // values
    for (long t = 0; t < s->Tv; ++t) {
      uint8_t *r, *vmask;
      if (rec_of(t, h, &r, &vmask)) return -2;
      const int tau = static_cast<int>(t % 16);
      const int w = tau / 8, b = (tau % 8) / 2, rr = tau % 2;
      static const int byte_of_tok[2][2] = {{0, 2}, {1, 3}};  // [w][r]
      for (int ch = 0; ch < d; ++ch) {
        const int mt = ch / 16, a = ch % 8, high = (ch % 16) / 8;
        const int L = 4 * a + b;
        const long off = VC + (mt / 4) * 512 + L * 16 + (mt % 4) * 4 + byte_of_tok[w][rr];
        put_nibble(r, vmask, off, high, s->vcode[h][t * d + ch]);
      }
      const int e = rr + 2 * w;
      for (int k = 0; k < 4; ++k) {
        put_f32(r, vmask, VM + ((2 * k) * 4 + b) * 16 + 4 * e, s->vs[h][t * 4 + k]);
        put_f32(r, vmask, VM + ((2 * k + 1) * 4 + b) * 16 + 4 * e, s->vmn[h][t * 4 + k]);
      }
    }
  }
  return 0;
}

// Residual rings: key ring [H][G][d], token t at row t mod G; value ring
// [H][R][d], token t at row t mod R. kvalid / vvalid flag the rows in use.
void orc_seq_ring_image(const orc_seq* s, uint16_t* kring, uint8_t* kvalid, uint16_t* vring,
                        uint8_t* vvalid) {
  const orc_cfg& c = s->cfg;
  const int H = c.num_kv_heads, d = c.head_dim, G = c.group_k, R = c.residual_v;
  for (int h = 0; h < H; ++h) {
    for (size_t i = 0; i < s->kres[h].size(); ++i) {
      const long t = s->Tk + static_cast<long>(i);
      const long row = t % G;
      std::memcpy(kring + (static_cast<long>(h) * G + row) * d, s->kres[h][i].data(), d * 2);
      if (kvalid) kvalid[h * G + row] = 1;
    }
    for (size_t i = 0; i < s->vres[h].size(); ++i) {
      const long t = s->Tv + static_cast<long>(i);
      const long row = t % R;
      std::memcpy(vring + (static_cast<long>(h) * R + row) * d, s->vres[h][i].data(), d * 2);
      if (vvalid) vvalid[h * R + row] = 1;
    }
  }
}

}  // extern "C"
