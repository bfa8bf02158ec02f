// ORACLE — test infrastructure only. Plain, slow, single-threaded CPU encoder
// for byte-level BPE, written from the method's description and sharing
// nothing with the CUDA encoder. Only tests, the smoke check and the bench's
// CPU-baseline leg may load it.
//
// It follows "Tokenization LLM: building an inference engine in C++"
// (glitch4techs), sections "Technical analysis" through "Vocabulary lookup":
//   1. pre-tokenize each document with the GPT-2-style split, given there by
//      its categories (contractions, words, numbers, punctuation, whitespace)
//      and the worked example "Hello world!" -> ["Hello", " world", "!"];
//      every piece is encoded on its own;
//   2. map every UTF-8 byte of a piece to its byte-to-unicode symbol (the
//      printable stand-in that lets every byte 0..255 be a vocabulary string;
//      byte 0xF0 maps to U+00F0);
//   3. repeat: list the adjacent symbol pairs, look each up in merge_rank,
//      take the lowest rank and merge that pair, until no ranked pair is left;
//   4. look every resulting symbol string up in the vocabulary.
// The two maps are the page's std::unordered_map vocabulary (string -> id) and
// unordered_map<pair<string, string>, int, PairHash> merge_rank.
//
// Readings where the pages leave a step open:
//   * The split is the six ordered alternatives
//       's|'t|'re|'ve|'m|'ll|'d | ?\p{L}+ | ?\p{N}+ | ?[^\s\p{L}\p{N}]+ |
//       \s+(?!\S) | \s+
//     tried in order at each position, each greedy with backtracking, as a
//     regex engine runs them. Letter = general category L*, number = N*,
//     whitespace = the White_Space property (unicode_ranges.inc).
//   * Invalid UTF-8: a lead byte followed by the right continuation bytes and
//     decoding to a scalar value (not overlong, not a surrogate, at most
//     U+10FFFF) is one codepoint; any other byte is a unit of its own that is
//     neither letter, number nor whitespace.
//   * One merge step replaces every occurrence of the chosen pair, scanning
//     left to right without overlap ("Tokenisierung": [a, a, a] with the merge
//     (a, a) becomes [aa, a]), and the next step looks at all pairs again.
//   * Rank = row index of the merge table; lower rank merges first.
// Parity pins for every step are in tests/test_oracle_pins.py.

#include <cstdint>
#include <cstring>
#include <string>
#include <utility>
#include <vector>
#include <unordered_map>

namespace {

// ------------------------------------------------------------ code points --

struct Range { uint32_t first, last; int cls; };
const Range kRanges[] = {
#include "unicode_ranges.inc"
};
const int kOther = 0, kLetter = 1, kNumber = 2, kSpace = 3;

int codepoint_class(int32_t cp) {
  if (cp < 0) return kOther;  // an invalid byte
  int lo = 0, hi = (int)(sizeof(kRanges) / sizeof(kRanges[0])) - 1;
  while (lo <= hi) {
    int mid = (lo + hi) / 2;
    if ((uint32_t)cp < kRanges[mid].first) hi = mid - 1;
    else if ((uint32_t)cp > kRanges[mid].last) lo = mid + 1;
    else return kRanges[mid].cls;
  }
  return kOther;
}

// Decode the unit that starts at s[p]: returns its byte length and sets cp
// (-1 for an invalid byte).
int decode_unit(const uint8_t* s, int64_t n, int64_t p, int32_t* cp) {
  uint8_t b = s[p];
  int len;
  uint32_t v;
  if (b < 0x80) { *cp = b; return 1; }
  if ((b & 0xE0) == 0xC0) { len = 2; v = b & 0x1F; }
  else if ((b & 0xF0) == 0xE0) { len = 3; v = b & 0x0F; }
  else if ((b & 0xF8) == 0xF0) { len = 4; v = b & 0x07; }
  else { *cp = -1; return 1; }
  if (p + len > n) { *cp = -1; return 1; }
  for (int k = 1; k < len; ++k) {
    uint8_t c = s[p + k];
    if ((c & 0xC0) != 0x80) { *cp = -1; return 1; }
    v = (v << 6) | (c & 0x3F);
  }
  const uint32_t min_for_len[5] = {0, 0, 0x80, 0x800, 0x10000};
  if (v < min_for_len[len] || v > 0x10FFFF || (v >= 0xD800 && v <= 0xDFFF)) { *cp = -1; return 1; }
  *cp = (int32_t)v;
  return len;
}

struct Unit { int64_t pos; int len; int32_t cp; int cls; };

std::vector<Unit> units_of(const uint8_t* s, int64_t n) {
  std::vector<Unit> u;
  for (int64_t p = 0; p < n;) {
    int32_t cp;
    int len = decode_unit(s, n, p, &cp);
    u.push_back({p, len, cp, codepoint_class(cp)});
    p += len;
  }
  return u;
}

// ------------------------------------------------------------- pre-tokenize --

// Each alternative returns the unit index where its match ends, or -1.
using Units = std::vector<Unit>;

int64_t alt_contraction(const Units& u, int64_t p) {
  int64_t n = (int64_t)u.size();
  if (u[p].cp != '\'') return -1;
  static const char* kSuffixes[] = {"s", "t", "re", "ve", "m", "ll", "d"};
  for (const char* suf : kSuffixes) {
    int64_t k = (int64_t)std::strlen(suf);
    if (p + k >= n) continue;
    bool ok = true;
    for (int64_t j = 0; j < k; ++j) ok = ok && u[p + 1 + j].cp == suf[j];
    if (ok) return p + 1 + k;
  }
  return -1;
}

bool in_class(const Unit& x, int want) {
  if (want == kOther) return x.cls == kOther;
  return x.cls == want;
}

// " ?X+" with X one of letter, number, other ([^\s\p{L}\p{N}]).
int64_t alt_optional_space_run(const Units& u, int64_t p, int want) {
  int64_t n = (int64_t)u.size();
  // First try with the optional space taken, then without it.
  if (u[p].cp == ' ' && p + 1 < n && in_class(u[p + 1], want)) {
    int64_t q = p + 1;
    while (q < n && in_class(u[q], want)) ++q;
    return q;
  }
  if (in_class(u[p], want)) {
    int64_t q = p;
    while (q < n && in_class(u[q], want)) ++q;
    return q;
  }
  return -1;
}

// "\s+(?!\S)": the longest whitespace run, giving back one unit at a time
// until the next unit is not a non-whitespace unit.
int64_t alt_space_not_before_nonspace(const Units& u, int64_t p) {
  int64_t n = (int64_t)u.size();
  if (u[p].cls != kSpace) return -1;
  int64_t q = p;
  while (q < n && u[q].cls == kSpace) ++q;
  for (int64_t end = q; end > p; --end) {
    bool next_is_nonspace = end < n && u[end].cls != kSpace;
    if (!next_is_nonspace) return end;
  }
  return -1;
}

int64_t alt_space(const Units& u, int64_t p) {
  int64_t n = (int64_t)u.size();
  if (u[p].cls != kSpace) return -1;
  int64_t q = p;
  while (q < n && u[q].cls == kSpace) ++q;
  return q;
}

int64_t match_at(const Units& u, int64_t p) {
  int64_t e;
  if ((e = alt_contraction(u, p)) >= 0) return e;
  if ((e = alt_optional_space_run(u, p, kLetter)) >= 0) return e;
  if ((e = alt_optional_space_run(u, p, kNumber)) >= 0) return e;
  if ((e = alt_optional_space_run(u, p, kOther)) >= 0) return e;
  if ((e = alt_space_not_before_nonspace(u, p)) >= 0) return e;
  if ((e = alt_space(u, p)) >= 0) return e;
  return p + 1;  // unreachable: every unit is matched by one alternative
}

// Byte offsets (relative to s) where the pieces of s start.
std::vector<int64_t> pretokenize(const uint8_t* s, int64_t n) {
  Units u = units_of(s, n);
  std::vector<int64_t> starts;
  for (int64_t p = 0; p < (int64_t)u.size();) {
    starts.push_back(u[p].pos);
    p = match_at(u, p);
  }
  return starts;
}

// ---------------------------------------------------------- byte to unicode --

// Bytes that are printable (33..126, 161..172, 174..255) stand for the
// codepoint of the same value; the remaining 68 bytes take 256, 257, ... in
// byte order.
struct ByteMap {
  int32_t to_cp[256];
  std::string to_str[256];
  std::unordered_map<int32_t, int> from_cp;
  ByteMap() {
    int next = 256;
    for (int b = 0; b < 256; ++b) {
      bool printable = (b >= 33 && b <= 126) || (b >= 161 && b <= 172) || (b >= 174 && b <= 255);
      to_cp[b] = printable ? b : next++;
      from_cp[to_cp[b]] = b;
      std::string& s = to_str[b];
      uint32_t c = (uint32_t)to_cp[b];
      if (c < 0x80) s.push_back((char)c);
      else { s.push_back((char)(0xC0 | (c >> 6))); s.push_back((char)(0x80 | (c & 0x3F))); }
    }
  }
};

const ByteMap& byte_map() {
  static ByteMap m;
  return m;
}

std::string symbols_of_bytes(const uint8_t* b, int64_t n) {
  std::string s;
  for (int64_t i = 0; i < n; ++i) s += byte_map().to_str[b[i]];
  return s;
}

// ------------------------------------------------------------------- model --

struct PairHash {
  size_t operator()(const std::pair<std::string, std::string>& p) const {
    size_t h1 = std::hash<std::string>()(p.first), h2 = std::hash<std::string>()(p.second);
    return h1 ^ (h2 + 0x9E3779B97F4A7C15ull + (h1 << 6) + (h1 >> 2));
  }
};

struct Oracle {
  std::unordered_map<std::string, int32_t> vocabulary;
  std::unordered_map<std::pair<std::string, std::string>, int64_t, PairHash> merge_rank;
  std::vector<std::string> id_to_string;
  std::string error;

  bool init(const int32_t* merges, int64_t n_merges, const uint8_t* vb, const int64_t* vo, int64_t n_vocab) {
    id_to_string.resize((size_t)n_vocab);
    for (int64_t id = 0; id < n_vocab; ++id) {
      std::string s = symbols_of_bytes(vb + vo[id], vo[id + 1] - vo[id]);
      id_to_string[(size_t)id] = s;
      if (s.empty()) continue;  // unused id
      if (!vocabulary.emplace(s, (int32_t)id).second) { error = "duplicate vocabulary string"; return false; }
    }
    for (int64_t k = 0; k < n_merges; ++k) {
      int32_t a = merges[3 * k], b = merges[3 * k + 1];
      if (a < 0 || b < 0 || a >= n_vocab || b >= n_vocab) { error = "merge id out of range"; return false; }
      auto key = std::make_pair(id_to_string[(size_t)a], id_to_string[(size_t)b]);
      if (!merge_rank.emplace(key, k).second) { error = "duplicate merge pair"; return false; }
    }
    return true;
  }

  // One pre-token: bytes -> symbols -> lowest-rank merge loop -> ids.
  bool encode_piece(const uint8_t* b, int64_t n, std::vector<int32_t>& out) {
    std::vector<std::string> sym;
    for (int64_t i = 0; i < n; ++i) sym.push_back(byte_map().to_str[b[i]]);
    for (;;) {
      int64_t best = -1;
      size_t at = 0;
      for (size_t i = 0; i + 1 < sym.size(); ++i) {
        auto it = merge_rank.find(std::make_pair(sym[i], sym[i + 1]));
        if (it != merge_rank.end() && (best < 0 || it->second < best)) { best = it->second; at = i; }
      }
      if (best < 0) break;
      std::string first = sym[at], second = sym[at + 1];
      std::vector<std::string> next;
      for (size_t i = 0; i < sym.size();) {
        if (i + 1 < sym.size() && sym[i] == first && sym[i + 1] == second) {
          next.push_back(first + second);
          i += 2;
        } else {
          next.push_back(sym[i]);
          i += 1;
        }
      }
      sym.swap(next);
    }
    for (const std::string& s : sym) {
      auto it = vocabulary.find(s);
      if (it == vocabulary.end()) { error = "symbol missing from vocabulary"; return false; }
      out.push_back(it->second);
    }
    return true;
  }
};

}  // namespace

extern "C" {

void* orc_new(const int32_t* merges, int64_t n_merges, const uint8_t* vocab_bytes,
              const int64_t* vocab_offsets, int64_t n_vocab) {
  Oracle* o = new Oracle();
  if (!o->init(merges, n_merges, vocab_bytes, vocab_offsets, n_vocab)) {
    delete o;
    return nullptr;
  }
  return o;
}

void orc_free(void* h) { delete (Oracle*)h; }

// Piece start offsets of one text (no document structure). Returns the count,
// or -(count) when cap is too small.
int64_t orc_pretokenize(const uint8_t* s, int64_t n, int64_t* starts, int64_t cap) {
  std::vector<int64_t> v = pretokenize(s, n);
  if ((int64_t)v.size() > cap) return -(int64_t)v.size();
  for (size_t i = 0; i < v.size(); ++i) starts[i] = v[i];
  return (int64_t)v.size();
}

// Start bits of a batch: bit i of bits (uint32 words) is set iff a piece
// starts at byte i; each document [doc_offsets[k], doc_offsets[k + 1]) is
// split on its own.
void orc_pretokenize_batch(const uint8_t* bytes, const int64_t* doc_offsets, int64_t n_docs, uint32_t* bits) {
  for (int64_t k = 0; k < n_docs; ++k) {
    int64_t a = doc_offsets[k], n = doc_offsets[k + 1] - a;
    for (int64_t st : pretokenize(bytes + a, n)) {
      int64_t i = a + st;
      bits[i >> 5] |= 1u << (i & 31);
    }
  }
}

// Decoded units of a text: writes (byte offset, codepoint or -1, class) rows.
int64_t orc_units(const uint8_t* s, int64_t n, int64_t* rows, int64_t cap) {
  Units u = units_of(s, n);
  if ((int64_t)u.size() > cap) return -(int64_t)u.size();
  for (size_t i = 0; i < u.size(); ++i) {
    rows[3 * i] = u[i].pos;
    rows[3 * i + 1] = u[i].cp;
    rows[3 * i + 2] = u[i].cls;
  }
  return (int64_t)u.size();
}

int32_t orc_class(int32_t cp) { return codepoint_class(cp); }
int32_t orc_byte_to_unicode(int32_t b) { return (b >= 0 && b < 256) ? byte_map().to_cp[b] : -1; }

// Encode one piece (no pre-tokenization); returns the number of ids.
int64_t orc_encode_piece(void* h, const uint8_t* s, int64_t n, int32_t* out, int64_t cap) {
  std::vector<int32_t> ids;
  if (!((Oracle*)h)->encode_piece(s, n, ids)) return -1;
  if ((int64_t)ids.size() > cap) return -2;
  for (size_t i = 0; i < ids.size(); ++i) out[i] = ids[i];
  return (int64_t)ids.size();
}

// Encode documents [first, first + count) of a batch. Document k is
// bytes[doc_offsets[k] .. doc_offsets[k + 1]). Writes ids and per-document
// offsets (count + 1 entries, starting at 0). Returns the number of ids, -1 on
// an error, -2 when cap is too small.
int64_t orc_encode_batch(void* h, const uint8_t* bytes, const int64_t* doc_offsets, int64_t first,
                         int64_t count, int32_t* out_ids, int64_t cap, int64_t* out_offsets) {
  Oracle* o = (Oracle*)h;
  std::vector<int32_t> ids;
  int64_t total = 0;
  out_offsets[0] = 0;
  for (int64_t k = first; k < first + count; ++k) {
    const uint8_t* d = bytes + doc_offsets[k];
    int64_t n = doc_offsets[k + 1] - doc_offsets[k];
    std::vector<int64_t> starts = pretokenize(d, n);
    for (size_t i = 0; i < starts.size(); ++i) {
      int64_t e = (i + 1 < starts.size()) ? starts[i + 1] : n;
      ids.clear();
      if (!o->encode_piece(d + starts[i], e - starts[i], ids)) return -1;
      if (total + (int64_t)ids.size() > cap) return -2;
      for (int32_t id : ids) out_ids[total++] = id;
    }
    out_offsets[k - first + 1] = total;
  }
  return total;
}

// Decode: the bytes of every id in order (symbol strings mapped back through
// the inverse byte-to-unicode map). Returns the byte count, -1 on an unknown
// id, -2 when cap is too small.
int64_t orc_decode(void* h, const int32_t* ids, int64_t n, uint8_t* out, int64_t cap) {
  Oracle* o = (Oracle*)h;
  int64_t w = 0;
  for (int64_t i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= (int64_t)o->id_to_string.size()) return -1;
    const std::string& s = o->id_to_string[(size_t)ids[i]];
    Units u = units_of((const uint8_t*)s.data(), (int64_t)s.size());
    for (const Unit& x : u) {
      auto it = byte_map().from_cp.find(x.cp);
      if (it == byte_map().from_cp.end()) return -1;
      if (w >= cap) return -2;
      out[w++] = (uint8_t)it->second;
    }
  }
  return w;
}

const char* orc_error(void* h) { return h ? ((Oracle*)h)->error.c_str() : "null handle"; }

}  // extern "C"
