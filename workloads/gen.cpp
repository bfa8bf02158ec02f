// Seeded synthetic inputs for batched byte-level BPE encoding.
//
// This file is input generation only. It draws corpora and documents, and it
// runs the BPE trainer that turns a corpus into a ranked merge table. Both the
// CUDA encoder and the CPU oracle consume what it produces as plain data; it
// holds none of the encoder's arithmetic (no pre-tokenizer predicate, no
// lowest-rank merge loop, no vocabulary lookup).
//
// Workload recipe (text generators):
//   * word list: 2,000 distinct lowercase words, lengths uniform in 2..9,
//     letters uniform in a..z; drawn by Zipf(s = 1.1) over word rank.
//   * ASCII token: 3% a run of 1..6 uniform digits, else a word; 5% of words
//     get a capital first letter, 4% a trailing char from .,!?'
//   * mixed-script token: 80% ASCII token, 10% a word of 2..9 letters from
//     U+00C0..U+00FF without U+00D7/U+00F7, 7% a run of 1..8 CJK ideographs
//     from U+4E00..U+9FFF, 3% one emoji from U+1F300..U+1F5FF.
//   * tokens are joined by single spaces; the long-context documents instead
//     end a line every 40..120 bytes with a newline plus 0..16 spaces.
//
// Trainer ("Tokenisierung", section "Byte Pair Encoding schrittweise"): count
// adjacent token pairs in the corpus, take the most frequent pair, on a tie
// the one with the smallest IDs (lexicographic on (left, right)), give it the
// next free ID, replace its occurrences left to right without overlap, and
// count again; stop after the requested number of merges or when no pair is
// left. Pairs are counted inside pre-tokens only, because a merge never
// crosses a pre-token ("Hugging Face Tokenizers v1", section on how v1 works).
//
// Randomness is splitmix64 (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014). Floating point uses only
// + - * / on doubles with contraction off, plus the series below for exp and
// log, so the same seed gives the same bytes on x86-64 and AArch64.

#include <cstdint>
#include <cstring>
#include <cmath>
#include <string>
#include <vector>
#include <unordered_map>
#include <queue>
#include <algorithm>

namespace {

struct Rng {
  uint64_t s;
  explicit Rng(uint64_t seed) : s(seed) {}
  uint64_t next() {
    uint64_t z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
  // uniform in [0, n)
  uint64_t below(uint64_t n) { return (uint64_t)(((__uint128_t)next() * n) >> 64); }
  // uniform in [lo, hi]
  int64_t range(int64_t lo, int64_t hi) { return lo + (int64_t)below((uint64_t)(hi - lo + 1)); }
  // uniform in [0, 1)
  double unit() { return (double)(next() >> 11) * (1.0 / 9007199254740992.0); }
};

uint64_t mix_seed(uint64_t a, uint64_t b) {
  Rng r(a ^ (b * 0xD1B54A32D192ED03ull));
  r.next();
  return r.next();
}

const double kLn2 = 0.69314718055994530942;

// log(x) for x > 0: x = m * 2^e with m in [sqrt(1/2), sqrt(2)), then
// log(m) = 2 atanh(t), t = (m - 1) / (m + 1), summed as a power series.
double det_log(double x) {
  int e = 0;
  double m = std::frexp(x, &e);  // exact
  if (m < 0.70710678118654752440) { m *= 2.0; e -= 1; }
  double t = (m - 1.0) / (m + 1.0);
  double t2 = t * t, term = t, sum = 0.0;
  for (int k = 1; k < 40; k += 2) { sum += term / (double)k; term *= t2; }
  return 2.0 * sum + (double)e * kLn2;
}

// exp(y): y = k ln2 + r with |r| <= ln2 / 2, Taylor series for exp(r).
double det_exp(double y) {
  double kf = y / kLn2;
  long k = (long)(kf < 0 ? kf - 0.5 : kf + 0.5);
  double r = y - (double)k * kLn2;
  double term = 1.0, sum = 1.0;
  for (int n = 1; n < 30; ++n) { term = term * r / (double)n; sum += term; }
  return std::ldexp(sum, (int)k);
}

// Standard normal by the Marsaglia polar method.
double normal(Rng& r) {
  for (;;) {
    double u = 2.0 * r.unit() - 1.0, v = 2.0 * r.unit() - 1.0;
    double s = u * u + v * v;
    if (s > 0.0 && s < 1.0) return u * std::sqrt(-2.0 * det_log(s) / s);
  }
}

void put_utf8(std::string& out, uint32_t cp) {
  if (cp < 0x80) {
    out.push_back((char)cp);
  } else if (cp < 0x800) {
    out.push_back((char)(0xC0 | (cp >> 6)));
    out.push_back((char)(0x80 | (cp & 0x3F)));
  } else if (cp < 0x10000) {
    out.push_back((char)(0xE0 | (cp >> 12)));
    out.push_back((char)(0x80 | ((cp >> 6) & 0x3F)));
    out.push_back((char)(0x80 | (cp & 0x3F)));
  } else {
    out.push_back((char)(0xF0 | (cp >> 18)));
    out.push_back((char)(0x80 | ((cp >> 12) & 0x3F)));
    out.push_back((char)(0x80 | ((cp >> 6) & 0x3F)));
    out.push_back((char)(0x80 | (cp & 0x3F)));
  }
}

struct Words {
  std::vector<std::string> words;
  std::vector<double> cdf;  // Zipf(1.1) cumulative weights over rank
  Words() {
    Rng r(0xB9E20000ull);
    std::unordered_map<std::string, int> seen;
    while (words.size() < 2000) {
      int len = (int)r.range(2, 9);
      std::string w;
      for (int i = 0; i < len; ++i) w.push_back((char)('a' + r.below(26)));
      if (seen.emplace(w, 1).second) words.push_back(w);
    }
    double acc = 0.0;
    for (int k = 1; k <= 2000; ++k) {
      acc += det_exp(-1.1 * det_log((double)k));
      cdf.push_back(acc);
    }
  }
  const std::string& zipf(Rng& r) const {
    double u = r.unit() * cdf.back();
    size_t i = (size_t)(std::upper_bound(cdf.begin(), cdf.end(), u) - cdf.begin());
    if (i >= words.size()) i = words.size() - 1;
    return words[i];
  }
};

const Words& words() {
  static Words w;
  return w;
}

void ascii_token(Rng& r, std::string& out) {
  if (r.unit() < 0.03) {
    int n = (int)r.range(1, 6);
    for (int i = 0; i < n; ++i) out.push_back((char)('0' + r.below(10)));
    return;
  }
  std::string w = words().zipf(r);
  if (r.unit() < 0.05) w[0] = (char)(w[0] - 'a' + 'A');
  out += w;
  if (r.unit() < 0.04) {
    static const char kPunct[] = ".,!?'";
    out.push_back(kPunct[r.below(5)]);
  }
}

void mixed_token(Rng& r, std::string& out) {
  double u = r.unit();
  if (u < 0.80) {
    ascii_token(r, out);
  } else if (u < 0.90) {
    int n = (int)r.range(2, 9);
    for (int i = 0; i < n; ++i) {
      uint32_t cp;
      do { cp = 0xC0 + (uint32_t)r.below(64); } while (cp == 0xD7 || cp == 0xF7);
      put_utf8(out, cp);
    }
  } else if (u < 0.97) {
    int n = (int)r.range(1, 8);
    for (int i = 0; i < n; ++i) put_utf8(out, 0x4E00 + (uint32_t)r.below(0x9FFF - 0x4E00 + 1));
  } else {
    put_utf8(out, 0x1F300 + (uint32_t)r.below(0x1F5FF - 0x1F300 + 1));
  }
}

// Cut s to at most n bytes without splitting a UTF-8 sequence.
void cut_at_codepoint(std::string& s, size_t n) {
  if (s.size() <= n) return;
  while (n > 0 && ((unsigned char)s[n] & 0xC0) == 0x80) --n;
  s.resize(n);
}

enum Script { kAscii = 0, kMixed = 1 };

// Tokens joined by single spaces until at least n bytes, then cut.
void text(Rng& r, Script script, size_t n, std::string& out, bool newlines) {
  size_t start = out.size();
  size_t line_start = out.size();
  int64_t line_len = newlines ? r.range(40, 120) : 0;
  bool first = true;
  while (out.size() - start < n) {
    if (!first) {
      if (newlines && (int64_t)(out.size() - line_start) >= line_len) {
        out.push_back('\n');
        line_start = out.size();
        int indent = (int)r.range(0, 16);
        out.append((size_t)indent, ' ');
        line_len = r.range(40, 120);
      } else {
        out.push_back(' ');
      }
    }
    first = false;
    if (script == kAscii) ascii_token(r, out); else mixed_token(r, out);
  }
  std::string tail = out.substr(start);
  cut_at_codepoint(tail, n);
  out.resize(start);
  out += tail;
}

// Configuration table. Sizes in bytes.
struct Cfg {
  Script corpus_script;
  int64_t corpus_bytes;
  int64_t n_merges;
  int64_t n_docs;
};

const Cfg kCfgs[6] = {
    {kAscii, 0, 0, 0},
    {kAscii, 256 << 10, 512, 256},          // 1 tiny
    {kMixed, 16 << 20, 32000, 16384},       // 2 mixed-script
    {kAscii, 64 << 20, 150000, 16},         // 3 long context
    {kAscii, 256 << 10, 512, 4096},         // 4 adversarial (uses the tiny table)
    {kAscii, 32 << 20, 100000, 4194304},    // 5 serving batch
};

void make_doc(int cfg, uint64_t seed, int64_t k, std::string& d) {
  Rng r(mix_seed(seed, (uint64_t)k));
  d.clear();
  switch (cfg) {
    case 1: text(r, kAscii, (size_t)r.range(1024, 4096), d, false); break;
    case 2: {
      double len = det_exp(det_log(4096.0) + 1.0 * normal(r));
      int64_t n = (int64_t)(len + 0.5);
      if (n < 1) n = 1;
      if (n > (16 << 20)) n = 16 << 20;
      text(r, kMixed, (size_t)n, d, false);
      break;
    }
    case 3: text(r, kMixed, (size_t)8 << 20, d, true); break;
    case 4: {
      int64_t run = r.range(1024, 65536);
      int64_t pick = r.range(0, 36);  // 26 letters, 10 digits, CJK
      std::string before, after, ws;
      text(r, kAscii, (size_t)(run / 18), before, false);
      std::string long_run;
      if (pick < 26) {
        long_run.assign((size_t)run, (char)('a' + pick));
      } else if (pick < 36) {
        long_run.assign((size_t)run, (char)('0' + pick - 26));
      } else {
        std::string one;
        put_utf8(one, 0x4E00 + (uint32_t)r.below(0x9FFF - 0x4E00 + 1));
        for (int64_t i = 0; i + 3 <= run; i += 3) long_run += one;
      }
      int64_t nws = r.range(1, 4096);
      static const char kWs[] = " \t\n";
      for (int64_t i = 0; i < nws; ++i) ws.push_back(kWs[r.below(3)]);
      text(r, kAscii, (size_t)(run / 18), after, false);
      d = before;
      d.push_back(' ');
      d += long_run;
      d += ws;
      d += after;
      break;
    }
    case 5: text(r, kAscii, (size_t)r.range(64, 448), d, false); break;
    default: break;
  }
}

// ---------------------------------------------------------------- trainer --

// Corpus split for the trainer. The corpora come from the generators above,
// whose alphabet is ASCII, Latin-1 letters, CJK ideographs and emoji joined by
// single spaces; for that alphabet a pre-token is an optional single space
// followed by a run of letters, a run of digits or a run of other symbols, or
// a run of whitespace.
int trainer_class(uint32_t cp) {
  if ((cp >= 'a' && cp <= 'z') || (cp >= 'A' && cp <= 'Z')) return 1;
  if (cp >= 0xC0 && cp <= 0xFF && cp != 0xD7 && cp != 0xF7) return 1;
  if (cp >= 0x4E00 && cp <= 0x9FFF) return 1;
  if (cp >= '0' && cp <= '9') return 2;
  if (cp == ' ' || (cp >= 9 && cp <= 13)) return 3;
  return 4;
}

struct Unit { int64_t pos; int len; int cls; };

std::vector<Unit> trainer_units(const uint8_t* s, int64_t n) {
  std::vector<Unit> u;
  for (int64_t p = 0; p < n;) {
    uint8_t b = s[p];
    int len = b < 0x80 ? 1 : b < 0xE0 ? 2 : b < 0xF0 ? 3 : 4;
    if (p + len > n) len = (int)(n - p);
    uint32_t cp = b;
    if (len == 2) cp = ((b & 0x1Fu) << 6) | (s[p + 1] & 0x3Fu);
    if (len == 3) cp = ((b & 0x0Fu) << 12) | ((s[p + 1] & 0x3Fu) << 6) | (s[p + 2] & 0x3Fu);
    if (len == 4) cp = ((b & 0x07u) << 18) | ((s[p + 1] & 0x3Fu) << 12) | ((s[p + 2] & 0x3Fu) << 6) | (s[p + 3] & 0x3Fu);
    u.push_back({p, len, trainer_class(cp)});
    p += len;
  }
  return u;
}

struct Trainer {
  std::vector<std::vector<int32_t>> words;
  std::vector<int64_t> freq;
  std::unordered_map<uint64_t, int64_t> count;
  std::unordered_map<uint64_t, std::vector<int32_t>> where;
  std::vector<int64_t> stamp;

  static uint64_t key(int32_t a, int32_t b) { return ((uint64_t)(uint32_t)a << 32) | (uint32_t)b; }

  struct Cand {
    int64_t c; int32_t a, b;
    bool operator<(const Cand& o) const {  // max-heap: larger count, then smaller (a, b)
      if (c != o.c) return c < o.c;
      if (a != o.a) return a > o.a;
      return b > o.b;
    }
  };
  std::priority_queue<Cand> pq;

  void pairs_of(const std::vector<int32_t>& s, std::vector<uint64_t>& out) {
    out.clear();
    for (size_t i = 0; i + 1 < s.size(); ++i) out.push_back(key(s[i], s[i + 1]));
    std::sort(out.begin(), out.end());
  }

  void add_pair(uint64_t k, int64_t delta, int32_t w, std::vector<uint64_t>* touched) {
    count[k] += delta;
    if (delta > 0) where[k].push_back(w);
    if (touched) touched->push_back(k);
  }

  int64_t run(int64_t n_merges, int32_t* out) {
    stamp.assign(words.size(), -1);
    std::vector<uint64_t> before, after;
    for (int32_t w = 0; w < (int32_t)words.size(); ++w) {
      pairs_of(words[w], after);
      for (uint64_t k : after) add_pair(k, freq[w], w, nullptr);
    }
    for (auto& kv : count) pq.push({kv.second, (int32_t)(kv.first >> 32), (int32_t)(uint32_t)kv.first});
    int64_t made = 0;
    std::vector<uint64_t> touched;
    while (made < n_merges && !pq.empty()) {
      Cand c = pq.top();
      pq.pop();
      uint64_t k = key(c.a, c.b);
      auto it = count.find(k);
      if (it == count.end() || it->second != c.c || c.c <= 0) continue;  // stale entry
      int32_t nid = 256 + (int32_t)made;
      out[3 * made + 0] = c.a;
      out[3 * made + 1] = c.b;
      out[3 * made + 2] = nid;
      touched.clear();
      std::vector<int32_t> ws = where[k];
      for (int32_t w : ws) {
        if (stamp[w] == made) continue;
        stamp[w] = made;
        auto& s = words[w];
        pairs_of(s, before);
        std::vector<int32_t> t;
        t.reserve(s.size());
        for (size_t i = 0; i < s.size();) {
          if (i + 1 < s.size() && s[i] == c.a && s[i + 1] == c.b) { t.push_back(nid); i += 2; }
          else { t.push_back(s[i]); i += 1; }
        }
        s.swap(t);
        pairs_of(s, after);
        // Apply only the difference between the old and new pair multisets.
        size_t i = 0, j = 0;
        while (i < before.size() || j < after.size()) {
          if (j == after.size() || (i < before.size() && before[i] < after[j])) {
            add_pair(before[i++], -freq[w], w, &touched);
          } else if (i == before.size() || after[j] < before[i]) {
            add_pair(after[j++], freq[w], w, &touched);
          } else {
            ++i; ++j;
          }
        }
      }
      where.erase(k);
      std::sort(touched.begin(), touched.end());
      touched.erase(std::unique(touched.begin(), touched.end()), touched.end());
      for (uint64_t t : touched) {
        auto ct = count.find(t);
        if (ct == count.end()) continue;
        if (ct->second <= 0) { count.erase(ct); continue; }
        pq.push({ct->second, (int32_t)(t >> 32), (int32_t)(uint32_t)t});
      }
      ++made;
    }
    return made;
  }
};

}  // namespace

extern "C" {

// Word list entry i (0 <= i < 2000) copied to out (NUL-terminated, <= 16 B).
int wl_word(int i, char* out) {
  if (i < 0 || i >= 2000) return -1;
  std::strcpy(out, words().words[i].c_str());
  return (int)words().words[i].size();
}

int64_t wl_cfg_corpus_bytes(int cfg) { return (cfg >= 1 && cfg <= 5) ? kCfgs[cfg].corpus_bytes : -1; }
int64_t wl_cfg_n_merges(int cfg) { return (cfg >= 1 && cfg <= 5) ? kCfgs[cfg].n_merges : -1; }
int64_t wl_cfg_n_docs(int cfg) { return (cfg >= 1 && cfg <= 5) ? kCfgs[cfg].n_docs : -1; }

// Corpus of exactly wl_cfg_corpus_bytes(cfg) bytes or fewer (cut at a code
// point) written to out; returns its length.
int64_t wl_corpus(int cfg, uint64_t seed, uint8_t* out, int64_t cap) {
  if (cfg < 1 || cfg > 5) return -1;
  Rng r(seed);
  std::string s;
  s.reserve((size_t)kCfgs[cfg].corpus_bytes + 64);
  text(r, kCfgs[cfg].corpus_script, (size_t)kCfgs[cfg].corpus_bytes, s, false);
  if ((int64_t)s.size() > cap) return -1;
  std::memcpy(out, s.data(), s.size());
  return (int64_t)s.size();
}

// Documents [k0, k0 + n) of configuration cfg. Pass out == nullptr to get the
// byte lengths only (lens[n]); then call again with out sized to their sum.
// Each document draws from its own stream, so any subset is reproducible.
int64_t wl_docs(int cfg, uint64_t seed, int64_t k0, int64_t n, int64_t* lens, uint8_t* out) {
  if (cfg < 1 || cfg > 5 || n < 0) return -1;
  std::vector<int64_t> off((size_t)n + 1, 0);
  if (out != nullptr) {
    for (int64_t i = 0; i < n; ++i) off[(size_t)i + 1] = off[(size_t)i] + lens[i];
  }
  int64_t total = 0;
  int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : total, bad)
  for (int64_t i = 0; i < n; ++i) {
    std::string d;
    make_doc(cfg, seed, k0 + i, d);
    if (out == nullptr) {
      lens[i] = (int64_t)d.size();
    } else {
      if ((int64_t)d.size() != lens[i]) { bad += 1; continue; }
      std::memcpy(out + off[(size_t)i], d.data(), d.size());
    }
    total += (int64_t)d.size();
  }
  return bad ? -1 : total;
}

}  // extern "C"

namespace {
// The trainer's words: the distinct pre-tokens of the corpus (first-seen
// order) as byte-symbol sequences, with how often each occurs.
void trainer_words(const uint8_t* corpus, int64_t n, std::vector<std::vector<int32_t>>& words,
                   std::vector<int64_t>& freq) {
  std::vector<Unit> u = trainer_units(corpus, n);
  std::unordered_map<std::string, int32_t> index;
  size_t i = 0;
  while (i < u.size()) {
    size_t j = i;
    if (u[i].cls == 3) {
      if (corpus[u[i].pos] == ' ' && i + 1 < u.size() && u[i + 1].cls != 3) {
        j = i + 1;
        int c = u[j].cls;
        while (j < u.size() && u[j].cls == c) ++j;
      } else {
        while (j < u.size() && u[j].cls == 3) ++j;
      }
    } else {
      int c = u[i].cls;
      while (j < u.size() && u[j].cls == c) ++j;
    }
    int64_t a = u[i].pos, b = (j < u.size()) ? u[j].pos : n;
    std::string w((const char*)corpus + a, (size_t)(b - a));
    auto it = index.find(w);
    if (it == index.end()) {
      index.emplace(w, (int32_t)words.size());
      std::vector<int32_t> syms;
      for (int64_t q = a; q < b; ++q) syms.push_back((int32_t)corpus[q]);
      words.push_back(std::move(syms));
      freq.push_back(1);
    } else {
      freq[(size_t)it->second] += 1;
    }
    i = j;
  }
}
}  // namespace

extern "C" {

// BPE trainer over a corpus: writes up to n_merges rows (left, right, new_id)
// to merges_out and returns the number of merges made.
int64_t wl_train(const uint8_t* corpus, int64_t n, int64_t n_merges, int32_t* merges_out) {
  Trainer t;
  trainer_words(corpus, n, t.words, t.freq);
  return t.run(n_merges, merges_out);
}

// The trainer's word list of a corpus: returns the number of words and sets
// *total_bytes; when bytes is non-null also writes the words' bytes back to
// back, offsets[n_words + 1] and counts[n_words] (size them from a first call
// with bytes == nullptr).
int64_t wl_train_words(const uint8_t* corpus, int64_t n, int64_t* total_bytes, uint8_t* bytes, int64_t* offsets,
                       int64_t* counts) {
  std::vector<std::vector<int32_t>> words;
  std::vector<int64_t> freq;
  trainer_words(corpus, n, words, freq);
  int64_t total = 0;
  for (const auto& w : words) total += (int64_t)w.size();
  *total_bytes = total;
  if (bytes) {
    int64_t at = 0;
    offsets[0] = 0;
    for (size_t k = 0; k < words.size(); ++k) {
      for (int32_t b : words[k]) bytes[at++] = (uint8_t)b;
      offsets[k + 1] = at;
      counts[k] = freq[k];
    }
  }
  return (int64_t)words.size();
}

// FNV-1a 64 over n bytes, continuing from state h (start with
// 0xcbf29ce484222325). A digest for comparing id streams, not part of any
// encoding: offset basis and prime are the published FNV-1a 64 parameters.
uint64_t wl_fnv1a64(const uint8_t* p, int64_t n, uint64_t h) {
  for (int64_t i = 0; i < n; ++i) {
    h ^= p[i];
    h *= 0x100000001b3ull;
  }
  return h;
}

}  // extern "C"
