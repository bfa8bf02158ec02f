// Batched byte-level BPE encoding on one GB300 (sm_103a): CUDA kernels and
// the C ABI declared in include/bpe_gb300.h.
//
// The method: glitch4techs, "Tokenization LLM: building an inference engine
// in C++", sections "Technical analysis" (GPT-2-style split; each piece is
// encoded on its own), "Byte-level encoding" (UTF-8 bytes, byte-level
// symbols), "Byte Pair Encoding algorithm" (repeat: lowest-rank adjacent pair
// merges, until none is left) and "Vocabulary lookup". Merges replace left to
// right without overlap (tokenwerk, "Tokenisierung", section "Byte Pair
// Encoding schrittweise").
//
// GPU design (none of it is on the pages, whose engines are CPU code):
//   * One pass over the input (k_tiles, tiles.cuh): a warp per 2016-byte tile
//     splits it, probes the word cache for every pre-token, and writes the
//     tile's ids to its stage slot, reserving room for the misses (their
//     byte length) and a placeholder for each pre-token over 64 bytes.
//   * Split (ascii_split32 in tiles.cuh, start_mask32 here): each lane takes
//     two words of 32 bytes.
//     - When they and their context are ASCII, carry-free SWAR range tests
//       give per-byte class masks, and the split rules are a dozen mask
//       operations; each apostrophe resolves its contraction in place.
//     - Otherwise a UTF-8 unit scan builds the same masks from a two-level
//       codepoint class table.
//     - Multi-byte whitespace falls back to the per-byte predicate
//       starts_piece.
//   * Symbols are token ids: byte b starts as byte_id[b]. An open-addressed
//     pair table of 32-byte buckets maps (left_id, right_id) to {rank,
//     new_id}. Because bytes(new_id) = bytes(left) || bytes(right) (checked
//     by bpe_build), the final symbols are the vocabulary ids.
//   * Word cache ("Hugging Face Tokenizers v1", section on word caching: the
//     same pre-token always gives the same ids, so a memo from pre-token bytes
//     to ids skips the merge loop).
//     - bpe_build fills it once, by running the merge loop on strings of 2 to
//       16 bytes: vocabulary strings, space-stripped vocabulary words and
//       prefixes of both.
//     - A pre-token found there takes the stored ids; one of a single byte is
//       its own token.
//   * Cache misses (at most 64 bytes) are merged GPU-wide (k_misses): a lane
//     per miss of up to 8 bytes (merge_thread), groups of 8, 16 or 32 lanes
//     for longer ones (merge_group: each step is a group-wide minimum, a
//     ballot of the pair's positions and a run-parity mask for the
//     non-overlapping left-to-right choice). memo.cuh adds a per-call memo of
//     repeated misses.
//   * Longer pre-tokens are merged by a whole CTA each (k_giants,
//     merge_long) in a device pool indexed by input byte, so each owns the
//     pool range of its own bytes.
//   * A scan of the tiles' final counts, then k_compact (ids into place
//     without the holes, document offsets) and k_giant_copy (the long
//     pre-tokens' ids). No kernel waits on another CTA.
//   * decode.cuh: ids back to bytes; train.cuh: the merge table trained on
//     the GPU.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <type_traits>
#include <unordered_set>
#include <vector>

#include "../../include/bpe_gb300.h"

#define BPE_CLASS_TABLE_STORAGE static __device__ const
#include "class_table.inc"

namespace {

// ---------------------------------------------------------------- constants --

constexpr int kThreads = 256;         // threads per CTA of the CTA-wide merge (k_giants)
constexpr int kHalo = 16;             // context bytes on each side of a split window
constexpr int kShortMax = 64;         // longest pre-token merged inside its tile (by a lane group)
constexpr int kCacheMaxLen = 16;      // longest pre-token looked up in the word cache
constexpr int kCacheMaxIds = 3;       // most ids a cache entry holds
constexpr int kLongPerThread = 4;     // elements per thread per round of the CTA merge
constexpr int kRound = kThreads * kLongPerThread;
constexpr uint32_t kReprobe = 0xFFFFFFFEu;              // pair rank still to be looked up
constexpr uint32_t kInf = 0xFFFFFFFFu;
constexpr uint32_t kNone = 0xFFFFFFFFu;
constexpr uint32_t kEmptySlot = 0xFFFFFFFFu;  // left id of an unused pair-table slot

static_assert(kShortMax <= 64 && kCacheMaxLen <= 16, "group merges hold 2 symbols per lane");

// device status bits
constexpr uint32_t kStBadInput = 1u;
constexpr uint32_t kStTimeout = 2u;
constexpr uint32_t kStInternal = 4u;
constexpr uint32_t kStCapacity = 8u;

enum Cls { kO = 0, kL = 1, kN = 2, kS = 3 };

// 32-bit hashing: odd multipliers combine the words, then a xor-shift /
// multiply finalizer (the "lowbias32" constants of Chris Wellons' hash
// prospector) spreads them over the low bits the tables index with.
__host__ __device__ inline uint32_t mix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x7FEB352Du;
  h ^= h >> 15;
  h *= 0x846CA68Bu;
  h ^= h >> 16;
  return h;
}

__host__ __device__ inline uint32_t pair_hash(uint32_t a, uint32_t b) {
  return mix32(a * 0x9E3779B1u + b * 0x85EBCA77u);
}

// Word cache key: the pre-token's bytes little-endian in x0..x3 (bytes 0..15),
// zero padded, plus its length.
__host__ __device__ inline uint32_t cache_hash(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3, uint32_t len) {
  return mix32(x0 * 0x9E3779B1u + x1 * 0x85EBCA77u + x2 * 0xC2B2AE3Du + x3 * 0x27D4EB2Fu + len);
}

struct Tables {
  const uint4* ht;         // 2 entries per 32-byte bucket: {left, right, rank, new_id}
  uint32_t hmask;          // buckets - 1
  const int32_t* mrows;    // [n_merges][3] (left, right, new)
  const int32_t* byte_id;  // [256]
};

// Word cache entry, two uint4: {k0 lo, k0 hi, k1 lo, k1 hi}, {meta, id0, id1,
// id2}; meta = len | count << 5 | 1 << 31, 0 for an empty slot.
struct Cache {
  const uint4* e;
  uint32_t mask;  // slots - 1
  int enabled;
};

struct DevSmall {
  uint32_t status;
  uint32_t pad;
  int64_t total;                     // ids of the call
  unsigned long long tile_ctr;       // tiles taken by k_tiles' warps
  unsigned long long n_misses;       // cache misses handed to k_misses
  unsigned long long n_giants;       // pre-tokens deferred to k_giants
  unsigned long long giant_ctr;      // deferred pre-tokens taken by k_giants' CTAs
  unsigned long long n_ranges;       // long runs of tiles for k_prep_long
};


// ------------------------------------------------------------ small helpers --

// Rank of the pair (a, b), kInf if it is not a merge; *nw gets the merged id.
// One 32-byte read-only load (a pair bucket or a word-cache entry; both
// tables are 32-byte aligned) as a single 256-bit access.
__device__ __forceinline__ void ldg32(const uint4* p, uint4& lo, uint4& hi) {
  asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
      : "l"(p));
}

__device__ __forceinline__ uint32_t lookup_pair(const Tables& T, uint32_t a, uint32_t b, uint32_t* nw) {
  uint32_t bucket = pair_hash(a, b) & T.hmask;
  for (uint32_t probe = 0; probe <= T.hmask; ++probe) {
    uint4 u, v;
    ldg32(T.ht + 2ull * bucket, u, v);
    if (u.x == a && u.y == b) {
      *nw = u.w;
      return u.z;
    }
    if (v.x == a && v.y == b) {
      *nw = v.w;
      return v.z;
    }
    if (u.x == kEmptySlot || v.x == kEmptySlot) return kInf;
    bucket = (bucket + 1) & T.hmask;
  }
  return kInf;
}

__device__ __forceinline__ uint32_t lookup_rank(const Tables& T, uint32_t a, uint32_t b) {
  uint32_t nw;
  return lookup_pair(T, a, b, &nw);
}



// The rest of lookup_pair once the home bucket {u, v} of (a, b) is loaded.
__device__ __forceinline__ uint32_t lookup_pair_from(const Tables& T, uint32_t a, uint32_t b, uint32_t bucket, uint4 u,
                                                     uint4 v, uint32_t* nw) {
  for (uint32_t probe = 0; probe <= T.hmask; ++probe) {
    if (u.x == a && u.y == b) {
      *nw = u.w;
      return u.z;
    }
    if (v.x == a && v.y == b) {
      *nw = v.w;
      return v.z;
    }
    if (u.x == kEmptySlot || v.x == kEmptySlot) return kInf;
    bucket = (bucket + 1) & T.hmask;
    ldg32(T.ht + 2ull * bucket, u, v);
  }
  return kInf;
}

// Two pair lookups with both home buckets in flight together; a pair with
// a == kNone is skipped (rank kInf).
__device__ __forceinline__ void lookup_pair2(const Tables& T, uint32_t a1, uint32_t b1, uint32_t a2, uint32_t b2,
                                             uint32_t* r1, uint32_t* w1, uint32_t* r2, uint32_t* w2) {
  const uint32_t k1 = pair_hash(a1, b1) & T.hmask, k2 = pair_hash(a2, b2) & T.hmask;
  uint4 u1 = make_uint4(0, 0, 0, 0), v1 = u1, u2 = u1, v2 = u1;
  if (a1 != kNone) {
    ldg32(T.ht + 2ull * k1, u1, v1);
  }
  if (a2 != kNone) {
    ldg32(T.ht + 2ull * k2, u2, v2);
  }
  *r1 = a1 != kNone ? lookup_pair_from(T, a1, b1, k1, u1, v1, w1) : kInf;
  *r2 = a2 != kNone ? lookup_pair_from(T, a2, b2, k2, u2, v2, w2) : kInf;
}

__device__ __forceinline__ int cp_class(uint32_t cp) {
  uint32_t blk = kClassL1[cp >> 8];
  uint32_t w = kClassL2[blk * 16 + ((cp & 255) >> 4)];
  return (int)((w >> ((cp & 15) * 2)) & 3);
}

__device__ __forceinline__ bool is_cont(uint32_t b) { return (b & 0xC0) == 0x80; }

// ------------------------------------------------------------- UTF-8 units --
// A unit is a well-formed UTF-8 sequence (Unicode's table of well-formed byte
// sequences) or, failing that, one byte on its own. Sequences do not cross a
// document edge: [lo, hi) is the document of the position asked about.

template <typename I>
__device__ __forceinline__ int seq_len(const uint8_t* w, I hi, I q) {
  uint32_t b0 = w[q];
  if (b0 < 0x80) return 1;
  if (b0 < 0xC2) return 0;
  if (b0 < 0xE0) return (q + 1 < hi && is_cont(w[q + 1])) ? 2 : 0;
  if (b0 < 0xF0) {
    if (q + 2 >= hi) return 0;
    uint32_t b1 = w[q + 1];
    uint32_t lo1 = (b0 == 0xE0) ? 0xA0 : 0x80, hi1 = (b0 == 0xED) ? 0x9F : 0xBF;
    return (b1 >= lo1 && b1 <= hi1 && is_cont(w[q + 2])) ? 3 : 0;
  }
  if (b0 < 0xF5) {
    if (q + 3 >= hi) return 0;
    uint32_t b1 = w[q + 1];
    uint32_t lo1 = (b0 == 0xF0) ? 0x90 : 0x80, hi1 = (b0 == 0xF4) ? 0x8F : 0xBF;
    return (b1 >= lo1 && b1 <= hi1 && is_cont(w[q + 2]) && is_cont(w[q + 3])) ? 4 : 0;
  }
  return 0;
}

// Start of the unit that holds byte p, and that unit's sequence length (0 for
// a lone invalid byte).
template <typename I>
__device__ __forceinline__ I unit_start_of(const uint8_t* w, I lo, I hi, I p, int* len) {
  if (is_cont(w[p])) {
    for (int k = 1; k <= 3 && p - k >= lo; ++k) {
      I q = p - k;
      if (!is_cont(w[q])) {
        int L = seq_len(w, hi, q);
        if (L > k) { *len = L; return q; }
        break;
      }
    }
    *len = 0;
    return p;
  }
  *len = seq_len(w, hi, p);
  return p;
}

template <typename I>
__device__ __forceinline__ int unit_class(const uint8_t* w, I q, int len) {
  uint32_t b0 = w[q];
  if (len == 0) return kO;
  if (len == 1) return cp_class(b0);
  uint32_t cp;
  if (len == 2) cp = ((b0 & 0x1Fu) << 6) | (w[q + 1] & 0x3Fu);
  else if (len == 3) cp = ((b0 & 0x0Fu) << 12) | ((w[q + 1] & 0x3Fu) << 6) | (w[q + 2] & 0x3Fu);
  else cp = ((b0 & 0x07u) << 18) | ((w[q + 1] & 0x3Fu) << 12) | ((w[q + 2] & 0x3Fu) << 6) | (w[q + 3] & 0x3Fu);
  return cp_class(cp);
}

template <typename I>
__device__ __forceinline__ int class_at(const uint8_t* w, I lo, I hi, I p) {
  int len;
  I q = unit_start_of(w, lo, hi, p, &len);
  return unit_class(w, q, len);
}

// ---------------------------------------------------------- pre-tokenizer --
// The GPT-2-style split tries, at each position, the ordered alternatives
//   's|'t|'re|'ve|'m|'ll|'d | ' '?L+ | ' '?N+ | ' '?O+ | S+(?!S) | S+
// (L letter, N number, S whitespace, O anything else). Its pieces are fixed
// by a predicate over a few neighbouring units, decided in this order for a
// unit start i inside a document (the document start always starts a piece):
//   B0 c[i-1] is an apostrophe that starts a piece, and c[i..] begins a
//      contraction suffix (s t m d re ve ll): no boundary;
//   B1 a contraction ends at i (its apostrophe starts a piece): boundary;
//   B2 c[i] in S: boundary iff c[i-1] not in S, or c[i+1] exists and is not
//      in S (the last whitespace before a non-space is split off);
//   B3 otherwise: no boundary after a U+0020 (the optional space joins the
//      run), boundary after other whitespace, else boundary iff the classes
//      L / N / O of c[i-1] and c[i] differ.
// An apostrophe at j starts a piece iff j is the document start or c[j-1] is
// a letter, a number or whitespace other than U+0020.

__device__ __forceinline__ bool is_stmd(uint32_t b) { return b == 's' || b == 't' || b == 'm' || b == 'd'; }
__device__ __forceinline__ bool is_suffix2(uint32_t a, uint32_t b) {
  return (a == 'r' && b == 'e') || (a == 'v' && b == 'e') || (a == 'l' && b == 'l');
}

template <typename I>
__device__ __forceinline__ bool apostrophe_starts_piece(const uint8_t* w, I lo, I hi, I j) {
  if (j == lo) return true;
  int c = class_at(w, lo, hi, j - 1);
  return c == kL || c == kN || (c == kS && w[j - 1] != ' ');
}

// The predicate, one position at a time (reference form of the mask paths).
template <typename I>
__device__ bool starts_piece(const uint8_t* w, I lo, I hi, I i) {
  if (i == lo) return true;
  int len;
  if (unit_start_of(w, lo, hi, i, &len) != i) return false;
  const int ci = unit_class(w, i, len);
  const uint32_t bp = w[i - 1];
  const int cprev = class_at(w, lo, hi, i - 1);
  if (bp == '\'') {  // B0
    const uint32_t b0 = w[i];
    const bool suffix = is_stmd(b0) || (i + 1 < hi && is_suffix2(b0, w[i + 1]));
    if (suffix && apostrophe_starts_piece(w, lo, hi, i - 1)) return false;
  }
  if (i - 2 >= lo && w[i - 2] == '\'' && is_stmd(bp) && apostrophe_starts_piece(w, lo, hi, i - 2)) return true;
  if (i - 3 >= lo && w[i - 3] == '\'' && is_suffix2(w[i - 2], bp) && apostrophe_starts_piece(w, lo, hi, i - 3))
    return true;
  if (ci == kS) {  // B2
    if (cprev != kS) return true;
    const I e = i + (len > 0 ? len : 1);
    return e < hi && class_at(w, lo, hi, e) != kS;
  }
  if (bp == ' ') return false;  // B3
  if (cprev == kS) return true;
  return ci != cprev;
}

// 0x80 in each byte of w (four ASCII bytes) that is a letter / digit /
// whitespace / U+0020, by carry-free range tests: for an ASCII byte x,
// x + (0x80 - lo) has bit 7 set iff x >= lo.
struct Ascii4 {
  uint32_t L, N, S, SP;
};

__device__ __forceinline__ Ascii4 ascii_classes(uint32_t w) {
  const uint32_t H = 0x80808080u;
  const uint32_t t = w | 0x20202020u;  // fold case
  Ascii4 r;
  r.L = (t + 0x1F1F1F1Fu) & ~(t + 0x05050505u) & H;   // 'a' .. 'z'
  r.N = (w + 0x50505050u) & ~(w + 0x46464646u) & H;   // '0' .. '9'
  const uint32_t y = w ^ 0x20202020u;
  r.SP = ~(y + 0x7F7F7F7Fu) & H;                      // == 0x20
  r.S = ((w + 0x77777777u) & ~(w + 0x72727272u) & H) | r.SP;  // 0x09 .. 0x0D or 0x20
  return r;
}

// SWAR class flags of four ASCII bytes (0x80 in each byte that is a letter,
// a digit, whitespace, or U+0020); bytes must be below 0x80 (no carries).
struct Flags4 {
  uint32_t L, N, S, SP;
};

__device__ __forceinline__ Flags4 ascii_flags(uint32_t w) {
  const uint32_t H = 0x80808080u;
  const uint32_t t = w | 0x20202020u;  // fold case
  Flags4 f;
  f.L = (t + 0x1F1F1F1Fu) & ~(t + 0x05050505u) & H;   // 'a' .. 'z'
  f.N = (w + 0x50505050u) & ~(w + 0x46464646u) & H;   // '0' .. '9'
  f.SP = ~((w ^ 0x20202020u) + 0x7F7F7F7Fu) & H;      // == 0x20
  f.S = ((w + 0x77777777u) & ~(w + 0x72727272u) & H) | f.SP;  // 0x09 .. 0x0D or 0x20
  return f;
}

// Eight 0x80 flags of words a, b -> 8 bits in byte order, in bits 24..31.
__device__ __forceinline__ uint32_t gather8(uint32_t a, uint32_t b) { return ((a >> 4) | b) * 0x00204081u; }
// 0x80-per-byte mask of a word -> 4 bits (byte j -> bit j).
__device__ __forceinline__ uint32_t movemask4(uint32_t m) { return ((m >> 7) * 0x01020408u) >> 24; }

// A 32-bit shared-memory load the compiler must issue as written, at the
// aligned word address given. The funnel shifts of adjacent words below read
// their words through this, so that no load of theirs can become a wider or
// shifted access. This is a guard, not a known fix: an earlier kernel that did
// the split and the encode in one CTA raised "misaligned address", and the
// cause was never found (a CPU emulation under address and undefined-behaviour
// checks was clean); a compiler-merged unaligned shared load was one suspect.
__device__ __forceinline__ uint32_t lds_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"((unsigned)__cvta_generic_to_shared(p)));
  return v;
}

// Asynchronous global-to-shared copy of 16 bytes (both addresses 16-byte
// aligned); a thread issues all of its copies before it waits for any.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((unsigned)__cvta_generic_to_shared(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }


// Bits [start, start + 32) of a shared bit array.
__device__ __forceinline__ uint32_t bits32_at(const uint32_t* bits, int start) {
  const int w = start >> 5, sh = start & 31;
  return __funnelshift_r(lds_u32(bits + w), lds_u32(bits + w + 1), sh);
}

}  // namespace

// ------------------------------------------------------------------ window --

namespace {

// A warp's scratch while its lanes merge pre-tokens in groups (merge_group).
struct GroupScratch {
  uint32_t sym[64], rank[64], nw[64];
};

// What the split needs: the window (CHUNK bytes whose start bits are computed,
// AFTER more, and kHalo bytes of context on each side) with its document-edge
// and outside-document bit masks, and room for the start bits.
template <int CHUNK, int AFTER, bool DOCS>
struct __align__(16) WindowSmem {
  static constexpr int kLen = kHalo + CHUNK + AFTER + kHalo;  // window bytes
  static constexpr int kWords = (kLen + 31) / 32;
  uint8_t win[kLen + 16];
  uint32_t docbits[DOCS ? kWords + 2 : 1];  // a document (or the area after the last one) starts here
  uint32_t outbits[kWords + 2];   // byte belongs to no document
  uint32_t startbits[(CHUNK + AFTER) / 32];
  int64_t chunk;
};

// Barrier of the kThreads threads of a CTA (named barrier 1).
__device__ __forceinline__ void cta_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

__device__ __forceinline__ bool bit_at(const uint32_t* bits, int i) { return (bits[i >> 5] >> (i & 31)) & 1u; }

// Document bounds [lo, hi) around window index i: the nearest document edge at
// or before i and the next one after i (at most kHalo away is all that is
// read), or the window edges.
template <class SS>
__device__ __forceinline__ void doc_bounds(const SS& S, int i, int* lo, int* hi) {
  int a = i;
  while (a > 0 && a > i - kHalo && !bit_at(S.docbits, a)) --a;
  *lo = a;
  int b = i + 1;
  while (b < SS::kLen && b <= i + kHalo && !bit_at(S.docbits, b)) ++b;
  *hi = b;
}

template <class SS>
__device__ __forceinline__ bool starts_piece_at(const SS& S, int i) {
  if (bit_at(S.outbits, i)) return false;
  int lo, hi;
  doc_bounds(S, i, &lo, &hi);
  return starts_piece<int>(S.win, lo, hi, i);
}

// Bits [start, start + 64) of a shared bit array.
__device__ __forceinline__ uint64_t bits64_at(const uint32_t* bits, int start) {
  const int w = start >> 5, sh = start & 31;
  const uint32_t a = lds_u32(bits + w), b = lds_u32(bits + w + 1), c = lds_u32(bits + w + 2);
  return (uint64_t)__funnelshift_r(a, b, sh) | (uint64_t)__funnelshift_r(b, c, sh) << 32;
}

// Boundary rules on class masks. Bit k of every mask is window byte
// p0 - 8 + k; the result is bits 8..39 (positions p0 .. p0 + 31). U marks unit
// starts, L / N / S the class of the unit holding each byte, SP bytes equal to
// U+0020, AP apostrophes, D document edges, O bytes outside every document.
// B2 and B3 come from the masks directly. Contractions (B0 / B1) are resolved
// per apostrophe: it starts a contraction when it is eligible (document start,
// or the unit before it is a letter, a number or whitespace other than
// U+0020) and the next one or two bytes of its document are a suffix; then
// the byte after it gets no boundary (B0) and the byte after the suffix gets
// one (B1).
// Contractions for the eligible apostrophes in cand (same bit layout): the
// byte after the apostrophe loses its boundary (B0) and the byte after the
// suffix gets one (B1).
template <class SS>
__device__ __forceinline__ uint64_t contractions(const SS& S, int p0, uint64_t cand, uint64_t D, uint64_t base) {
  uint64_t B0 = 0, B1 = 0;
  while (cand) {
    const int k = __ffsll((long long)cand) - 1;
    cand &= cand - 1;
    const int q = p0 - 8 + k;
    const uint32_t b1 = S.win[q + 1];
    if (is_stmd(b1)) {
      B0 |= 1ull << (k + 1);
      B1 |= 1ull << (k + 2);
    } else if (!((D >> (k + 2)) & 1u) && is_suffix2(b1, S.win[q + 2])) {
      B0 |= 1ull << (k + 1);
      B1 |= 1ull << (k + 3);
    }
  }
  return (base & ~B0) | B1;
}

constexpr uint64_t kApostropheBits = 0x7FFFFFFFE0ull;  // apostrophes at bytes p0 - 3 .. p0 + 30 matter

template <class SS>
__device__ __forceinline__ uint32_t boundaries32(const SS& S, int p0, uint64_t U, uint64_t L, uint64_t N,
                                                 uint64_t Sm, uint64_t SP, uint64_t AP, uint64_t D, uint64_t O) {
  const uint64_t Sp = Sm << 1, Lp = L << 1, Np = N << 1, SPp = SP << 1;
  const uint64_t Sn = Sm >> 1, Dn = D >> 1;
  const uint64_t B2 = Sm & (~Sp | (~Sn & ~Dn));
  const uint64_t B3 = ~Sm & ~SPp & (Sp | (L ^ Lp) | (N ^ Np));
  uint64_t base = D | B2 | B3;
  const uint64_t prev_ok = (L | N | (Sm & ~SP)) << 1;  // bit k: byte k - 1 makes an apostrophe at k eligible
  const uint64_t cand = AP & kApostropheBits & (D | prev_ok) & ~(D >> 1);
  if (cand) base = contractions(S, p0, cand, D, base);
  return (uint32_t)((U & ~O & base) >> 8);
}

// The same rules for bytes p0 - 4 .. p0 + 35 read as ASCII (word m of w32 =
// bytes p0 - 4 + 4 m), computed per byte on 0x80-per-byte masks (a byte's
// neighbours are a funnel shift away) and turned into bits once:
// base = D | X | B3 | (Y & ~Dn) with X = S & ~Sp and Y = S & ~Sn the two
// halves of B2, and C the apostrophes whose previous byte makes them
// eligible. *any gets the OR of the ten words: the result holds only if none
// has a byte >= 0x80.
template <class SS>
__device__ __forceinline__ uint32_t ascii_starts32(const SS& S, int p0, const uint32_t* w32, uint64_t D, uint64_t O,
                                                   uint32_t* any) {
  uint32_t wv[10];
#pragma unroll
  for (int m = 0; m < 10; ++m) wv[m] = lds_u32(w32 + m);
  Ascii4 prev = ascii_classes(wv[0]), cur = ascii_classes(wv[1]);
  uint32_t all = wv[0] | wv[1];
  // eligible apostrophes of word 0 (bytes p0 - 3 .. p0 - 1 are the ones used)
  uint32_t e_prev = prev.L | prev.N | (prev.S & ~prev.SP);
  const uint32_t c0 = movemask4(~((wv[0] ^ 0x27272727u) + 0x7F7F7F7Fu) & 0x80808080u & __funnelshift_l(0u, e_prev, 8));
  uint32_t z = 0, y = 0, c = 0, zlo = 0, ylo = 0, clo = 0;
#pragma unroll
  for (int m = 1; m <= 8; ++m) {
    all |= wv[m + 1];
    const Ascii4 next = ascii_classes(wv[m + 1]);
    const uint32_t Sp = __funnelshift_l(prev.S, cur.S, 8), Lp = __funnelshift_l(prev.L, cur.L, 8),
                   Np = __funnelshift_l(prev.N, cur.N, 8), SPp = __funnelshift_l(prev.SP, cur.SP, 8),
                   Sn = __funnelshift_r(cur.S, next.S, 8);
    const uint32_t B3 = ~cur.S & ~SPp & (Sp | (cur.L ^ Lp) | (cur.N ^ Np));
    const uint32_t Z = (cur.S & ~Sp) | B3, Y = cur.S & ~Sn;
    const uint32_t E = cur.L | cur.N | (cur.S & ~cur.SP);
    const uint32_t C = ~((wv[m] ^ 0x27272727u) + 0x7F7F7F7Fu) & 0x80808080u & __funnelshift_l(e_prev, E, 8);
    e_prev = E;
    if (m & 1) {
      zlo = Z >> 7;
      ylo = Y >> 7;
      clo = C >> 7;
    } else {
      // bytes of words m - 1 and m: bits 0..3 and 4..7 of the product's top
      // byte (the other partial products stay below bit 24), placed in byte
      // (m - 2) / 2 of the result
      const int i = (m - 2) / 2;
      const uint32_t sel = (0x3210u & ~(0xFu << (4 * i))) | (7u << (4 * i));
      z = __byte_perm(z, (zlo | (Z >> 3)) * 0x01020408u, sel);
      y = __byte_perm(y, (ylo | (Y >> 3)) * 0x01020408u, sel);
      c = __byte_perm(c, (clo | (C >> 3)) * 0x01020408u, sel);
    }
    prev = cur;
    cur = next;
  }
  *any = all;
  uint32_t base = (uint32_t)(D >> 8) | z | (y & ~(uint32_t)(D >> 9));
  // Contractions: eligible apostrophes, and apostrophes at a document start;
  // none followed by a document start.
  uint64_t cand = ((uint64_t)c << 8) | ((uint64_t)c0 << 4);
  uint64_t dap = D & kApostropheBits;
  while (dap) {
    const int k = __ffsll((long long)dap) - 1;
    dap &= dap - 1;
    if (S.win[p0 - 8 + k] == 0x27u) cand |= 1ull << k;
  }
  cand &= kApostropheBits & ~(D >> 1);
  if (cand) base = (uint32_t)(contractions(S, p0, cand, D, (uint64_t)base << 8) >> 8);
  return base & ~(uint32_t)(O >> 8);
}

// Start bits of window positions [p0, p0 + 32), p0 a multiple of 16.
template <class SS>
__device__ uint32_t start_mask32(const SS& S, int p0, bool try_ascii = true) {
  const uint64_t D = bits64_at(S.docbits, p0 - 8), O = bits64_at(S.outbits, p0 - 8);
  if ((uint32_t)(O >> 8) == 0xFFFFFFFFu) return 0;
  // Ten aligned window words: bytes p0 - 4 .. p0 + 35. ASCII: every byte is a
  // unit (skipped when the caller has already found a byte above 0x7F).
  if (try_ascii) {
    uint32_t any;
    const uint32_t ascii = ascii_starts32(S, p0, reinterpret_cast<const uint32_t*>(S.win + p0) - 1, D, O, &any);
    if (!(any & 0x80808080u)) return ascii;
  }
  // General: the UTF-8 units of bytes [p0 - 7, p0 + 33); each byte carries
  // its unit's class (bit k of the masks is byte p0 - 8 + k). Units starting
  // before p0 - 8 may be misread only up to p0 - 5, and nothing before p0 - 4
  // is used. ASCII bytes are units of their own, classed by the SWAR tests of
  // twelve aligned words with every byte above 0x7F cleared first; only the
  // bytes above 0x7F are walked, a unit at a time.
  const int base = p0 - 8;
  const uint32_t* w32 = reinterpret_cast<const uint32_t*>(S.win + base);
  uint64_t Lm = 0, Nm = 0, Sm = 0, SPm = 0, APm = 0, NA = 0;
#pragma unroll
  for (int i = 0; i < 6; ++i) {
    uint32_t wa = lds_u32(w32 + 2 * i), wb = lds_u32(w32 + 2 * i + 1);
    const uint32_t ha = wa & 0x80808080u, hb = wb & 0x80808080u;
    wa &= ~((ha >> 7) * 0xFFu);  // bytes above 0x7F -> 0 (class O, no apostrophe)
    wb &= ~((hb >> 7) * 0xFFu);
    const Flags4 fa = ascii_flags(wa), fb = ascii_flags(wb);
    const uint32_t xa = wa ^ 0x27272727u, xb = wb ^ 0x27272727u;
    const uint32_t aa = ~(xa + 0x7F7F7F7Fu) & 0x80808080u, ab = ~(xb + 0x7F7F7F7Fu) & 0x80808080u;
    const int sh = 8 * i;
    Lm |= (uint64_t)(gather8(fa.L, fb.L) >> 24) << sh;
    Nm |= (uint64_t)(gather8(fa.N, fb.N) >> 24) << sh;
    Sm |= (uint64_t)(gather8(fa.S, fb.S) >> 24) << sh;
    SPm |= (uint64_t)(gather8(fa.SP, fb.SP) >> 24) << sh;
    APm |= (uint64_t)(gather8(aa, ab) >> 24) << sh;
    NA |= (uint64_t)(gather8(ha, hb) >> 24) << sh;
  }
  const uint64_t kSpan = 0x1FFFFFFFFFEull;  // bits 1 .. 40
  uint64_t cons = 0, MBS = 0;                // continuation bytes of multi-byte units; multi-byte whitespace
  uint64_t na = NA & kSpan;
  while (na) {
    const int k = __ffsll((long long)na) - 1;
    na &= na - 1;
    if ((cons >> k) & 1ull) continue;  // inside the unit before
    const int q = base + k;
    const uint32_t dn = (uint32_t)(D >> (k + 1)) & 7u;  // document edges at q + 1 .. q + 3
    const int hi = dn ? q + __ffs(dn) : q + 4;
    const int len = seq_len(S.win, hi, q);
    const int cls = unit_class(S.win, q, len);
    const uint64_t unit = ((len > 1 ? (1ull << len) : 2ull) - 1ull) << k;  // its bytes
    if (len > 1) cons |= unit & ~(1ull << k);
    if (cls == kL) Lm |= unit;
    if (cls == kN) Nm |= unit;
    if (cls == kS) {
      Sm |= unit;
      if (len > 1) MBS |= 1ull << k;
    }
  }
  const uint64_t U = kSpan & ~cons;
  Lm &= kSpan;
  Nm &= kSpan;
  Sm &= kSpan;
  SPm &= kSpan;
  APm &= kSpan;
  uint32_t res = boundaries32(S, p0, U, Lm, Nm, Sm, SPm, APm, D, O);
  // Whitespace of several bytes (B2 looks past the whole unit): the per-byte
  // predicate.
  uint32_t fix = (uint32_t)(MBS >> 8);
  while (fix) {
    const int k = __ffs(fix) - 1;
    fix &= fix - 1;
    const uint32_t bit = 1u << k;
    res = (res & ~bit) | (starts_piece_at(S, p0 + k) ? bit : 0u);
  }
  return res;
}

// ----------------------------------------------------------- block helpers --

// Minimum over the CTA (two barriers; red is free again on return).
__device__ uint32_t block_min(uint32_t v, uint32_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
  if (lane == 0) red[warp] = v;
  cta_sync();
  uint32_t r = red[0];
  for (int k = 1; k < kThreads / 32; ++k) r = min(r, red[k]);
  cta_sync();
  return r;
}

// ----------------------------------------------------------- merge: short --
// One thread, symbols and pair ranks in memory it owns. rk[k] is the rank of
// (sym[k], sym[k+1]). A step takes the lowest rank, replaces every occurrence
// of that pair left to right without overlap, and re-probes only the pairs
// that touch a new symbol.

__device__ int merge_short(uint32_t* sym, uint32_t* rk, const uint8_t* src, int n, const Tables& T,
                           const int32_t* byte_id) {
  for (int k = 0; k < n; ++k) sym[k] = (uint32_t)byte_id[src[k]];
  if (n < 2) return n;
  for (int k = 0; k + 1 < n; ++k) rk[k] = lookup_rank(T, sym[k], sym[k + 1]);
  for (;;) {
    uint32_t best = kInf;
    for (int k = 0; k + 1 < n; ++k) best = min(best, rk[k]);
    if (best == kInf) break;
    const uint32_t nw = (uint32_t)T.mrows[3 * best + 2];
    int w = 0, prev_old = -1, k = 0;
    while (k < n) {
      uint32_t s;
      int old;
      if (k + 1 < n && rk[k] == best) {
        s = nw;
        old = -1;
        k += 2;
      } else {
        s = sym[k];
        old = k;
        k += 1;
      }
      if (w > 0) {
        uint32_t r = (old >= 0 && prev_old >= 0 && old == prev_old + 1) ? rk[prev_old] : lookup_rank(T, sym[w - 1], s);
        rk[w - 1] = r;
      }
      sym[w] = s;
      prev_old = old;
      ++w;
    }
    n = w;
    if (n < 2) break;
  }
  return n;
}

// ------------------------------------------------------ merge: lane group --
// G lanes of a warp (G = 8 or 32) merge one pre-token of n <= 2 G symbols
// together. Lane g holds positions g and g + G: the symbol, and the rank and
// merged id of the pair that starts there. A step takes the group's lowest
// rank and marks every position where that pair starts. Two marks are
// adjacent only when both symbols of the pair are equal; a left-to-right scan
// without overlap then keeps the first mark of each such run and every second
// one after it, which is computed for all positions at once from the run
// starts (bit masks of up to 64 positions). The merged symbols are written
// compacted to the warp's scratch and only the pairs that touch a merged
// symbol are looked up again. All 32 lanes call this together; a group with
// n == 0 idles. The final ids go to out[0 .. count).
template <int G>
__device__ uint32_t merge_group(GroupScratch& W, const uint8_t* src, uint32_t n, const Tables& T,
                                const int32_t* byte_id, uint32_t* out) {
  static_assert(G == 4 || G == 8 || G == 16 || G == 32, "group of 4, 8, 16 or 32 lanes");
  const int lane = threadIdx.x & 31;
  const int g = lane & (G - 1);
  const int goff = lane & ~(G - 1);
  const uint32_t gbits = G == 32 ? 0xFFFFFFFFu : ((1u << G) - 1u);
  uint32_t* ws = W.sym + (lane / G) * 2 * G;
  uint32_t* wr = W.rank + (lane / G) * 2 * G;
  uint32_t* ww = W.nw + (lane / G) * 2 * G;
  const uint32_t p0 = (uint32_t)g, p1 = (uint32_t)(g + G);

  uint32_t s0 = p0 < n ? (uint32_t)byte_id[src[p0]] : kNone;
  uint32_t s1 = p1 < n ? (uint32_t)byte_id[src[p1]] : kNone;
  ws[p0] = s0;
  ws[p1] = s1;
  __syncwarp();
  // masks of the group's positions: 32 bits while they fit
  using Mask = typename std::conditional<(2 * G <= 32), uint32_t, uint64_t>::type;
  constexpr int kMaskBits = 8 * (int)sizeof(Mask);
  uint32_t w0 = 0, w1 = 0;
  uint32_t r0 = p0 + 1 < n ? lookup_pair(T, s0, ws[p0 + 1], &w0) : kInf;
  uint32_t r1 = p1 + 1 < n ? lookup_pair(T, s1, ws[p1 + 1], &w1) : kInf;
  uint32_t cnt = n;
  for (;;) {
    uint32_t best = min(r0, r1);
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) best = min(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
    const bool go = best != kInf;
    if (!__any_sync(0xFFFFFFFFu, go)) break;
    const bool o0 = go && r0 == best, o1 = go && r1 == best;
    const uint32_t b0 = (__ballot_sync(0xFFFFFFFFu, o0) >> goff) & gbits;
    const uint32_t b1 = (__ballot_sync(0xFFFFFFFFu, o1) >> goff) & gbits;
    const Mask M = (Mask)b0 | ((Mask)b1 << G);
    const uint32_t any = b0 | b1;
    const uint32_t nwb = __shfl_sync(0xFFFFFFFFu, o0 ? w0 : w1, goff + (any ? __ffs(any) - 1 : 0));
    const Mask E = (Mask)0x5555555555555555ull;  // even positions
    const Mask run_start = M & ~(M << 1);
    const Mask even_runs = M & ~(M + (run_start & E));  // runs that start at an even position
    const Mask take = (even_runs & E) | (M & ~even_runs & ~E);
    const Mask valid = cnt >= (uint32_t)kMaskBits ? ~(Mask)0 : (((Mask)1 << cnt) - 1);
    const Mask keep = valid & ~(take << 1);
    __syncwarp();  // every lane has read the scratch before it is rewritten
    if (go) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t p = h ? p1 : p0;
        if ((keep >> p) & 1) {
          const uint32_t ni = (uint32_t)__popcll((uint64_t)(keep & (((Mask)1 << p) - 1)));
          const bool tp = (take >> p) & 1;
          const uint32_t q = tp ? p + 2 : p + 1;  // next kept position
          const bool tq = q < (uint32_t)kMaskBits && ((take >> q) & 1);
          ws[ni] = tp ? nwb : (h ? s1 : s0);
          wr[ni] = (tp || tq) ? kReprobe : (h ? r1 : r0);
          ww[ni] = h ? w1 : w0;
        }
      }
      cnt = (uint32_t)__popcll((uint64_t)keep);
    }
    __syncwarp();
    if (go) {  // a finished group keeps its registers
      s0 = p0 < cnt ? ws[p0] : kNone;
      s1 = p1 < cnt ? ws[p1] : kNone;
      r0 = p0 + 1 < cnt ? wr[p0] : kInf;
      r1 = p1 + 1 < cnt ? wr[p1] : kInf;
      w0 = ww[p0];
      w1 = ww[p1];
      if (r0 == kReprobe) r0 = lookup_pair(T, s0, ws[p0 + 1], &w0);
      if (r1 == kReprobe) r1 = lookup_pair(T, s1, ws[p1 + 1], &w1);
    }
  }
  if (p0 < cnt) out[p0] = s0;
  if (p1 < cnt) out[p1] = s1;
  return cnt;
}

// ------------------------------------------------------------ merge: long --
// The whole CTA merges one long pre-token in place in scr (the pool range of
// its own bytes, read and written in rounds of kRound elements; a round
// writes only below where it read). A step is one pass: the chosen pair
// (A, B) is replaced left to right without overlap, and every pair of the
// new sequence is looked up for the next step's lowest rank (four home
// buckets in flight a thread). The first pass merges nothing, so it only
// maps bytes to symbols and looks up their pairs, without scans or barriers. Within a round each thread takes
// kLongPerThread elements; whether its first element was consumed by the
// merge before it, and where its kept symbols go, come from one CTA scan of
// (transfer function, kept count) elements.

struct LongScratch {
  uint32_t* sym;   // [2][kRound]: a round's kept symbols (by round parity)
  uint32_t* red;   // [2][kThreads / 32]
  uint32_t* mred;  // [kThreads / 32]
};

// One scan element: bit 0 = "next element consumed" after this part when
// the part's first element was not consumed, bit 1 = the same when it was;
// bits 2..12 and 13..23 = symbols the part keeps in either case.
__device__ __forceinline__ uint32_t tfc_then(uint32_t a, uint32_t b) {
  const uint32_t a0 = a & 1u, a1 = (a >> 1) & 1u;
  const uint32_t b0 = (b >> 2) & 0x7FFu, b1 = (b >> 13) & 0x7FFu;
  const uint32_t f = ((b >> a0) & 1u) | ((b >> a1) & 1u) << 1;
  const uint32_t c0 = ((a >> 2) & 0x7FFu) + (a0 ? b1 : b0);
  const uint32_t c1 = ((a >> 13) & 0x7FFu) + (a1 ? b1 : b0);
  return f | c0 << 2 | c1 << 13;
}
constexpr uint32_t kTfcIdentity = 2u;
static_assert(kRound < 2048, "round counts fit in 11 bits");

__device__ uint32_t merge_long(const uint8_t* g_bytes, int64_t s, uint32_t n, int32_t* scr, const Tables& T,
                               const int32_t* byte_id, LongScratch L) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t len = n;
  bool first_pass = true;
  uint32_t A = kNone, B = kNone, NW = 0;  // the pair of this pass (none in the first)
  uint32_t par = 0;
  for (;;) {
    uint32_t W = 0, carry = 0, prev_sym = kNone, local_min = kInf;
    if (first_pass) {
      // Nothing merges in the first pass: every byte's symbol stays where it
      // is, so a thread looks up its own pairs (the next thread's first
      // symbol read directly) with no scan and no barrier.
      for (uint32_t r0 = 0; r0 < len; r0 += kRound) {
        uint32_t x[kLongPerThread + 1], bk[kLongPerThread];
        uint4 u[kLongPerThread], v[kLongPerThread];
        const uint32_t i0 = r0 + (uint32_t)tid * kLongPerThread;
#pragma unroll
        for (int k = 0; k <= kLongPerThread; ++k) x[k] = i0 + k < len ? (uint32_t)byte_id[g_bytes[s + i0 + k]] : kNone;
#pragma unroll
        for (int k = 0; k < kLongPerThread; ++k) {
          if (x[k] != kNone) scr[i0 + k] = (int32_t)x[k];
          bk[k] = pair_hash(x[k], x[k + 1]) & T.hmask;
          if (x[k + 1] != kNone) ldg32(T.ht + 2ull * bk[k], u[k], v[k]);
        }
#pragma unroll
        for (int k = 0; k < kLongPerThread; ++k) {
          if (x[k + 1] == kNone) continue;
          uint32_t nw;
          local_min = min(local_min, lookup_pair_from(T, x[k], x[k + 1], bk[k], u[k], v[k], &nw));
        }
      }
      W = len;
    }
    for (uint32_t r0 = 0; !first_pass && r0 < len; r0 += kRound, par ^= 1u) {
      uint32_t x[kLongPerThread + 1];
#pragma unroll
      for (int k = 0; k <= kLongPerThread; ++k) {
        const uint32_t idx = r0 + (uint32_t)tid * kLongPerThread + (uint32_t)k;
        x[k] = kNone;
        if (idx < len) x[k] = first_pass ? (uint32_t)byte_id[g_bytes[s + idx]] : (uint32_t)scr[idx];
      }
      bool hit[kLongPerThread];  // (x[k], x[k + 1]) is the pair of this pass
#pragma unroll
      for (int k = 0; k < kLongPerThread; ++k) hit[k] = !first_pass && x[k] == A && x[k + 1] == B;
      // this thread's part for both inputs: consumed out, symbols kept
      uint32_t e = 0;
#pragma unroll
      for (uint32_t in = 0; in < 2; ++in) {
        uint32_t consumed = in, kept = 0;
#pragma unroll
        for (int k = 0; k < kLongPerThread; ++k) {
          if (x[k] == kNone) break;
          if (consumed) {
            consumed = 0;
          } else {
            ++kept;
            consumed = hit[k];
          }
        }
        e |= consumed << in | kept << (in ? 13 : 2);
      }
      // CTA scan of the parts, one barrier
      uint32_t incl = e;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl = tfc_then(o, incl);
      }
      uint32_t* red = L.red + par * (kThreads / 32);
      if (lane == 31) red[warp] = incl;
      cta_sync();
      // every warp scans the warp totals on its first kThreads / 32 lanes
      uint32_t wt = lane < kThreads / 32 ? red[lane] : kTfcIdentity;
#pragma unroll
      for (int d = 1; d < kThreads / 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, wt, d);
        if (lane >= d) wt = tfc_then(o, wt);
      }
      const uint32_t all = __shfl_sync(0xFFFFFFFFu, wt, kThreads / 32 - 1);
      uint32_t before = __shfl_sync(0xFFFFFFFFu, wt, (warp + 31) & 31);
      if (warp == 0) before = kTfcIdentity;
      uint32_t ex = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
      if (lane == 0) ex = kTfcIdentity;
      before = tfc_then(before, ex);
      uint32_t consumed = (before >> carry) & 1u;
      uint32_t pos = carry ? (before >> 13) & 0x7FFu : (before >> 2) & 0x7FFu;
      const uint32_t round_cnt = carry ? (all >> 13) & 0x7FFu : (all >> 2) & 0x7FFu;
      carry = (all >> carry) & 1u;
      // the kept symbols, in order (a buffer per round parity, so the next
      // round's writes need no barrier after this round's reads)
      uint32_t* st_sym = L.sym + par * kRound;
#pragma unroll
      for (int k = 0; k < kLongPerThread; ++k) {
        if (x[k] == kNone) break;
        if (consumed) {
          consumed = 0;
        } else if (hit[k]) {
          st_sym[pos++] = NW;
          consumed = 1;
        } else {
          st_sym[pos++] = x[k];
        }
      }
      cta_sync();
      // the round's pairs (q - 1, q), kLongPerThread per thread with their
      // home buckets loaded together
      {
        uint32_t lf[kLongPerThread], rt[kLongPerThread], bk[kLongPerThread];
        uint4 u[kLongPerThread], v[kLongPerThread];
#pragma unroll
        for (int k = 0; k < kLongPerThread; ++k) {
          const uint32_t q = (uint32_t)tid + (uint32_t)k * kThreads;
          lf[k] = kNone;
          rt[k] = 0;
          if (q < round_cnt) {
            lf[k] = q == 0 ? prev_sym : st_sym[q - 1];
            rt[k] = st_sym[q];
            scr[W + q] = (int32_t)rt[k];
          }
          bk[k] = pair_hash(lf[k], rt[k]) & T.hmask;
          if (lf[k] != kNone) ldg32(T.ht + 2ull * bk[k], u[k], v[k]);
        }
#pragma unroll
        for (int k = 0; k < kLongPerThread; ++k) {
          if (lf[k] == kNone) continue;
          uint32_t nw;
          local_min = min(local_min, lookup_pair_from(T, lf[k], rt[k], bk[k], u[k], v[k], &nw));
        }
      }
      if (round_cnt > 0) prev_sym = st_sym[round_cnt - 1];
      W += round_cnt;
    }
    len = W;
    first_pass = false;
    const uint32_t best = block_min(local_min, L.mred);
    if (best == kInf) break;
    A = (uint32_t)T.mrows[3 * best];
    B = (uint32_t)T.mrows[3 * best + 1];
    NW = (uint32_t)T.mrows[3 * best + 2];
  }
  cta_sync();
  return len;
}

// Word-cache key of a short pre-token (window positions [kHalo + st, + len)):
// its bytes as four little-endian words, zero past len, read with aligned
// 32-bit shared loads and funnel shifts.
// A pre-token's cache key words: its bytes little-endian in x0..x3, zero
// padded (the length travels separately).
struct CacheKey {
  uint32_t x0, x1, x2, x3;
};


__device__ __forceinline__ uint32_t cache_slot(const CacheKey& K, uint32_t len, const Cache& C) {
  return cache_hash(K.x0, K.x1, K.x2, K.x3, len) & C.mask;
}


}  // namespace

#include "tiles.cuh"
#include "memo.cuh"
#include "decode.cuh"
#include "train.cuh"

namespace {

// Word-cache values: the ids of each string, computed by the same merge loop
// the encoder runs. out[4 i] = count, out[4 i + 1 .. 3] = first three ids.
__global__ void k_cache_values(const uint8_t* strs, const int64_t* offs, int64_t n, Tables T, uint32_t* out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  uint32_t sym[kCacheMaxLen], rk[kCacheMaxLen];
  const int len = (int)(offs[i + 1] - offs[i]);
  if (len < 1 || len > kCacheMaxLen) {
    out[4 * i] = 0;
    return;
  }
  const int cnt = merge_short(sym, rk, strs + offs[i], len, T, T.byte_id);
  out[4 * i] = (uint32_t)cnt;
  for (int q = 0; q < kCacheMaxIds; ++q) out[4 * i + 1 + q] = q < cnt ? sym[q] : 0u;
}

// x[0..n) += delta (document offsets of one slice of a host batch: to the
// slice's bytes before encoding, to the whole batch's ids after).
__global__ void k_offsets_shift(int64_t* x, int64_t n, int64_t delta) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    x[i] += delta;
}

// The call's token count into page-locked host memory, written by the GPU:
// a copy on the encode stream would queue behind the large downloads on the
// same copy engine and hold up the next slice's kernels.
__global__ void k_total_to_host(const DevSmall* small, int64_t* h_dst) {
  if (threadIdx.x == 0) *reinterpret_cast<volatile int64_t*>(h_dst) = small->total;
}

// ------------------------------------------------------------------- host --

thread_local std::string g_err;

int fail(int code, const std::string& msg) {
  g_err = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(BPE_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define CK(call)                                        \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    cudaGetDevice(&cur);
    if (prev >= 0 && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

struct bpe_handle {
  int device = 0;
  int n_sms = 1;  // multiprocessors of the device (grids of persistent kernels)
  int64_t n_merges = 0, n_vocab = 0;
  int monotone = 1;  // every merge's operands are made by lower ranks (bpe_merges_monotone)
  uint4* d_ht = nullptr;
  uint32_t hmask = 0;
  int32_t* d_mrows = nullptr;
  int32_t* d_byte_id = nullptr;
  uint8_t* d_vbytes = nullptr;
  int64_t* d_voffs = nullptr;
  uint4* d_vent = nullptr;  // per token: its first 12 bytes and its length (decoding)
  uint4* d_cache = nullptr;
  uint32_t cache_mask = 0;
  int64_t cache_entries = 0;
  int cache_enabled = 1;
  int call_memo = BPE_MEMO_AUTO;  // bpe_set_call_memo
  DevSmall* d_small = nullptr;
  DevSmall* h_small = nullptr;  // pinned
  void* d_ws = nullptr;
  size_t ws_bytes = 0;
  bool smem_set = false;
  cudaEvent_t ev_start = nullptr, ev_stop = nullptr;
  cudaEvent_t* ev_phase = nullptr;  // BPE_ENCODE_LAUNCHES + 1 caller-owned events, or null
  // bpe_encode_batch_host: kHostSlots slots of device buffers, copy streams,
  // events
  static constexpr int kHostSlots = 4;
  struct HostSlot {
    uint8_t* bytes = nullptr;
    int64_t* offs = nullptr;
    int32_t* ids = nullptr;
    int64_t* out_offs = nullptr;
    cudaEvent_t in = nullptr, done = nullptr, free = nullptr;
  } slot[kHostSlots];
  int64_t slot_bytes = 0, slot_docs = 0;  // capacity of each slot
  cudaStream_t s_h2d = nullptr, s_d2h = nullptr;
  int64_t* h_totals = nullptr;  // pinned, one per slice
  int64_t* d_totals = nullptr;  // the same memory as the device addresses it
  int64_t h_totals_cap = 0;
};

namespace {

int ensure_ws(bpe_handle* h, size_t need) {
  if (need <= h->ws_bytes) return BPE_OK;
  size_t sz = need + need / 4 + 4096;
  if (h->d_ws) CK(cudaFree(h->d_ws));
  h->d_ws = nullptr;
  h->ws_bytes = 0;
  CK(cudaMalloc(&h->d_ws, sz));
  h->ws_bytes = sz;
  return BPE_OK;
}

int read_status(bpe_handle* h, cudaStream_t st, DevSmall* out) {
  CK(cudaMemcpyAsync(h->h_small, h->d_small, sizeof(DevSmall), cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  *out = *h->h_small;
  if (out->status) CK(cudaMemsetAsync(&h->d_small->status, 0, sizeof(uint32_t), st));
  return BPE_OK;
}

int status_code(uint32_t s) {
  if (s & kStBadInput) return fail(BPE_ERR_BAD_INPUT, "offsets not monotone or outside the buffer, or an id out of range");
  if (s & kStTimeout) return fail(BPE_ERR_TIMEOUT, "a device-side wait gave up");
  if (s & kStCapacity) return fail(BPE_ERR_CAPACITY, "output capacity exceeded");
  if (s & kStInternal) return fail(BPE_ERR_INTERNAL, "device-side consistency check failed");
  return BPE_OK;
}

// Word cache: the ids of every vocabulary string of 2..16 bytes, of every
// vocabulary string that starts with a space with that space removed (the
// same word at the start of a line or document), and of every prefix of
// those (a word cut off by the end of a document), computed on the device by
// the merge loop, laid out as an open-addressed table (load at most 1/16,
// linear probing, keys of lower ids inserted first).
int build_word_cache(bpe_handle* h, const uint8_t* vocab_bytes, const int64_t* vocab_offsets, int64_t n_vocab) {
  std::vector<uint8_t> strs;
  std::vector<int64_t> offs{0};
  std::vector<uint64_t> prio;  // insertion order: a lower id (an earlier merge, a more frequent pair) first
  std::unordered_set<std::string> keys;
  // Single bytes are left out: a one-byte pre-token is its own token.
  auto add = [&](const uint8_t* b, int64_t L, uint64_t p) {
    if (L < 2 || L > kCacheMaxLen || !keys.insert(std::string((const char*)b, (size_t)L)).second) return;
    strs.insert(strs.end(), b, b + L);
    offs.push_back((int64_t)strs.size());
    prio.push_back(p);
  };
  for (int64_t id = 0; id < n_vocab; ++id)
    add(vocab_bytes + vocab_offsets[id], vocab_offsets[id + 1] - vocab_offsets[id], (uint64_t)id << 2);
  for (int64_t id = 0; id < n_vocab; ++id) {
    const int64_t L = vocab_offsets[id + 1] - vocab_offsets[id];
    if (L >= 2 && vocab_bytes[vocab_offsets[id]] == ' ')
      add(vocab_bytes + vocab_offsets[id] + 1, L - 1, (uint64_t)id << 2 | 1u);
  }
  // Prefixes of all of the above (a word cut off by the end of a document).
  for (int64_t i = 0, n0 = (int64_t)offs.size() - 1; i < n0; ++i) {
    const std::string w(strs.begin() + offs[i], strs.begin() + offs[i + 1]);  // copy: add() grows strs
    const uint64_t p = (prio[(size_t)i] & ~3ull) | 2u;
    for (size_t L = 2; L < w.size(); ++L) add(reinterpret_cast<const uint8_t*>(w.data()), (int64_t)L, p);
  }
  const int64_t n = (int64_t)offs.size() - 1;
  uint8_t* d_strs = nullptr;
  int64_t* d_offs = nullptr;
  uint32_t* d_out = nullptr;
  std::vector<uint32_t> vals((size_t)std::max<int64_t>(1, n) * 4);
  cudaError_t e = cudaSuccess;
  if (n > 0) {
    e = cudaMalloc(&d_strs, strs.size());
    if (e == cudaSuccess) e = cudaMalloc(&d_offs, offs.size() * sizeof(int64_t));
    if (e == cudaSuccess) e = cudaMalloc(&d_out, (size_t)n * 4 * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemcpy(d_strs, strs.data(), strs.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(d_offs, offs.data(), offs.size() * sizeof(int64_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) {
      Tables T{h->d_ht, h->hmask, h->d_mrows, h->d_byte_id};
      k_cache_values<<<(unsigned)((n + 127) / 128), 128>>>(d_strs, d_offs, n, T, d_out);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpy(vals.data(), d_out, (size_t)n * 4 * sizeof(uint32_t), cudaMemcpyDeviceToHost);
    cudaFree(d_strs);
    cudaFree(d_offs);
    cudaFree(d_out);
    if (e != cudaSuccess) return cuda_fail(e, "word cache values");
  }
  int64_t keep = 0;
  for (int64_t i = 0; i < n; ++i) keep += (vals[4 * i] >= 1 && vals[4 * i] <= (uint32_t)kCacheMaxIds);
  // Load at most 1/16, keys inserted by priority: a probe that meets another
  // key at the home slot costs its whole warp a second round trip, so the
  // keys of frequent pre-tokens should own their home slots.
  uint64_t slots = 16;
  while (slots < (uint64_t)keep * 16) slots <<= 1;
  std::vector<int64_t> order((size_t)n);
  for (int64_t i = 0; i < n; ++i) order[(size_t)i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int64_t x, int64_t y) { return prio[(size_t)x] < prio[(size_t)y]; });
  std::vector<uint4> table(slots * 2, make_uint4(0, 0, 0, 0));
  for (const int64_t i : order) {
    const uint32_t cnt = vals[4 * i];
    if (cnt < 1 || cnt > (uint32_t)kCacheMaxIds) continue;
    const uint32_t len = (uint32_t)(offs[i + 1] - offs[i]);
    uint64_t k0 = 0, k1 = 0;
    for (uint32_t q = 0; q < len; ++q) {
      const uint64_t b = strs[(size_t)offs[i] + q];
      if (q < 8) k0 |= b << (8 * q);
      else k1 |= b << (8 * (q - 8));
    }
    uint64_t slot =
        cache_hash((uint32_t)k0, (uint32_t)(k0 >> 32), (uint32_t)k1, (uint32_t)(k1 >> 32), len) & (slots - 1);
    while (table[slot * 2 + 1].x != 0) slot = (slot + 1) & (slots - 1);
    table[slot * 2] = make_uint4((uint32_t)k0, (uint32_t)(k0 >> 32), (uint32_t)k1, (uint32_t)(k1 >> 32));
    table[slot * 2 + 1] = make_uint4(len | (cnt << 5) | (1u << 31), vals[4 * i + 1], vals[4 * i + 2], vals[4 * i + 3]);
  }
  CK(cudaMalloc(&h->d_cache, table.size() * sizeof(uint4)));
  CK(cudaMemcpy(h->d_cache, table.data(), table.size() * sizeof(uint4), cudaMemcpyHostToDevice));
  h->cache_mask = (uint32_t)(slots - 1);
  h->cache_entries = keep;
  return BPE_OK;
}

}  // namespace

// -------------------------------------------------------- encode workspace --
// Regions of the per-call workspace, each starting on a 256-byte boundary:
// per tile its first document, record, first pre-token start and offset;
// the scan's block sums; the stage slots; the miss queue; the deferred-piece
// records; the long runs of k_prep_docs; the pool of the deferred pieces (an
// int32 per input byte).
namespace {
constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsSizes {
  size_t first_doc, rec, first_start, tile_base, block_sum, stage, misses, giants, ranges, pool, memo, follow, total;
  int64_t n_tiles, miss_cap, giant_cap, range_cap;
  uint64_t memo_slots;
};

constexpr uint64_t kMemoMaxSlots = uint64_t(1) << 24;  // the per-call memo's table: at most 128 MiB

// memo: room for the per-call memo of the misses (the table and the
// follower of each queue entry)
constexpr WsSizes ws_sizes(int64_t n_bytes, bool memo = false) {
  WsSizes z{};
  z.n_tiles = n_bytes / kTileOwn + 1;
  z.miss_cap = n_bytes / 2 + 64;  // a miss has at least 2 bytes
  z.giant_cap = n_bytes / (kShortMax + 1) + z.n_tiles + 16;
  z.range_cap = z.n_tiles / kPrepSpan + 16;
  z.first_doc = align256((size_t)z.n_tiles * sizeof(int64_t));
  z.rec = align256((size_t)z.n_tiles * sizeof(TileRec));
  z.first_start = align256((size_t)z.n_tiles * sizeof(int64_t));
  z.tile_base = align256((size_t)z.n_tiles * sizeof(uint64_t));
  z.block_sum = align256((size_t)(z.n_tiles / kScanThreads + 1) * sizeof(uint64_t));
  z.stage = align256((size_t)z.n_tiles * kTileBits * sizeof(uint32_t));
  z.misses = align256((size_t)z.miss_cap * sizeof(uint64_t));
  z.giants = align256((size_t)z.giant_cap * sizeof(GiantRec));
  z.ranges = align256((size_t)z.range_cap * sizeof(PrepRange));
  z.pool = align256((size_t)(n_bytes + 4) * sizeof(int32_t));
  z.memo_slots = 0;
  z.memo = z.follow = 0;
  if (memo) {
    z.memo_slots = 1024;
    while (z.memo_slots < kMemoMaxSlots && z.memo_slots < 2 * (uint64_t)z.miss_cap) z.memo_slots <<= 1;
    z.memo = align256(z.memo_slots * sizeof(uint64_t));
    z.follow = align256((size_t)z.miss_cap * sizeof(uint32_t));
  }
  z.total = z.first_doc + z.rec + z.first_start + z.tile_base + z.block_sum + z.stage + z.misses + z.giants +
            z.ranges + z.pool + z.memo + z.follow;
  return z;
}

struct Ws {
  int64_t n_tiles, miss_cap, giant_cap, range_cap;
  int64_t* first_doc;
  TileRec* rec;
  int64_t* first_start;
  uint64_t* tile_base;
  uint64_t* block_sum;
  uint32_t* stage;
  uint64_t* misses;
  GiantRec* giants;
  PrepRange* ranges;
  int32_t* pool;
  uint64_t* memo;   // null: no per-call memo
  uint32_t* follow;
  uint64_t memo_slots;
};

Ws ws_carve(unsigned char* base, int64_t n_bytes, bool memo = false) {
  const WsSizes z = ws_sizes(n_bytes, memo);
  Ws w;
  w.n_tiles = z.n_tiles;
  w.miss_cap = z.miss_cap;
  w.giant_cap = z.giant_cap;
  w.range_cap = z.range_cap;
  auto take = [&](size_t n) {
    unsigned char* p = base;
    base += n;
    return p;
  };
  w.first_doc = reinterpret_cast<int64_t*>(take(z.first_doc));
  w.rec = reinterpret_cast<TileRec*>(take(z.rec));
  w.first_start = reinterpret_cast<int64_t*>(take(z.first_start));
  w.tile_base = reinterpret_cast<uint64_t*>(take(z.tile_base));
  w.block_sum = reinterpret_cast<uint64_t*>(take(z.block_sum));
  w.stage = reinterpret_cast<uint32_t*>(take(z.stage));
  w.misses = reinterpret_cast<uint64_t*>(take(z.misses));
  w.giants = reinterpret_cast<GiantRec*>(take(z.giants));
  w.ranges = reinterpret_cast<PrepRange*>(take(z.ranges));
  w.pool = reinterpret_cast<int32_t*>(take(z.pool));
  w.memo = memo ? reinterpret_cast<uint64_t*>(take(z.memo)) : nullptr;
  w.follow = memo ? reinterpret_cast<uint32_t*>(take(z.follow)) : nullptr;
  w.memo_slots = z.memo_slots;
  return w;
}

// k_tiles' dynamic shared memory above the 48 KB default, once per device.
int tiles_smem_setup() {
  if (cudaFuncSetAttribute(k_tiles, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTileSmemBytes) != cudaSuccess)
    return fail(BPE_ERR_CUDA, "cudaFuncSetAttribute(k_tiles) failed");
  return BPE_OK;
}

// The per-call kernels on stream st: k_prep_docs, k_prep_long, k_tiles,
// k_misses, k_giants (which returns at once when nothing was deferred), the
// scan, k_compact and k_giant_copy (which returns at once when nothing was
// deferred). ev_start / ev_stop (may be null) bracket all of them; ev_phase
// (may be null) gets one event before the first and one after each.
int launch_encode(bpe_handle* h, const Ws& w, const uint8_t* d_bytes, int64_t n_bytes, const int64_t* d_doc_offsets,
                  int64_t n_docs, int32_t* d_out_ids, int64_t out_capacity, int64_t* d_out_offsets, cudaStream_t st,
                  cudaEvent_t ev_start, cudaEvent_t ev_stop, cudaEvent_t* ev_phase);
}  // namespace

// ---------------------------------------------- fixed scratch of the no-alloc encode --
// bpe_encode_batch_noalloc keeps its workspace in one array of static device
// memory per device, sized for kNoAllocMaxBytes input bytes.
namespace {
constexpr int64_t kNoAllocMaxBytes = int64_t(4) << 20;
constexpr size_t kNoAllocScratchBytes = ws_sizes(kNoAllocMaxBytes).total;
static_assert(kNoAllocScratchBytes < (size_t(64) << 20), "the fixed scratch stays below 64 MiB");
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_base[kNoAllocMaxDevices] = {};

// Once per device, with that device current: the scratch address and the
// tile kernel's shared-memory opt-in. Later calls only read the table.
int noalloc_setup(int dev, unsigned char** base) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return fail(BPE_ERR_INVALID_ARG, "bpe_encode_batch_noalloc: device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_base[dev]) {
    void* p = nullptr;
    CK(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    if (reinterpret_cast<uintptr_t>(p) & 255u)
      return fail(BPE_ERR_INTERNAL, "bpe_encode_batch_noalloc: scratch not 256-byte aligned");
    if (tiles_smem_setup()) return BPE_ERR_CUDA;
    g_noalloc_base[dev] = static_cast<unsigned char*>(p);
  }
  *base = g_noalloc_base[dev];
  return BPE_OK;
}
}  // namespace

namespace {
int launch_encode(bpe_handle* h, const Ws& w, const uint8_t* d_bytes, int64_t n_bytes, const int64_t* d_doc_offsets,
                  int64_t n_docs, int32_t* d_out_ids, int64_t out_capacity, int64_t* d_out_offsets, cudaStream_t st,
                  cudaEvent_t ev_start, cudaEvent_t ev_stop, cudaEvent_t* ev_phase) {
  if (ev_start) CK(cudaEventRecord(ev_start, st));
  int phase = 0;  // bpe_set_phase_events
  if (ev_phase) CK(cudaEventRecord(ev_phase[phase++], st));
  const int64_t n_tiles = w.n_tiles;
  const int prep_blocks = (int)std::min<int64_t>(4096, (n_docs + 2) / 256 + 1);
  k_prep_docs<<<prep_blocks, 256, 0, st>>>(d_doc_offsets, n_docs, n_bytes, n_tiles, w.first_doc, w.ranges,
                                           w.range_cap, h->d_small);
  CK(cudaGetLastError());
  if (ev_phase) CK(cudaEventRecord(ev_phase[phase++], st));
  k_prep_long<<<(unsigned)std::min<int64_t>(2 * h->n_sms, w.range_cap), 256, 0, st>>>(w.ranges, w.range_cap,
                                                                                    w.first_doc, n_tiles, h->d_small);
  CK(cudaGetLastError());
  if (ev_phase) CK(cudaEventRecord(ev_phase[phase++], st));
  TileArgs a;
  a.bytes = d_bytes;
  a.n_bytes = n_bytes;
  a.doc_offsets = d_doc_offsets;
  a.n_docs = n_docs;
  a.T = Tables{h->d_ht, h->hmask, h->d_mrows, h->d_byte_id};
  a.C = Cache{h->d_cache, h->cache_mask, h->cache_enabled && h->d_cache != nullptr};
  a.first_doc = w.first_doc;
  a.rec = w.rec;
  a.first_start = w.first_start;
  a.stage = w.stage;
  a.misses = w.misses;
  a.miss_cap = w.miss_cap;
  a.giants = w.giants;
  a.giant_cap = w.giant_cap;
  a.small = h->d_small;
  a.n_tiles = n_tiles;
  const int64_t grid = std::min<int64_t>((int64_t)kTileCtasPerSm * h->n_sms, (n_tiles + kTileWarps - 1) / kTileWarps);
  k_tiles<<<(unsigned)grid, kTileThreads, kTileSmemBytes, st>>>(a);
  CK(cudaGetLastError());
  if (ev_phase) CK(cudaEventRecord(ev_phase[phase++], st));
  if (w.memo) {  // the per-call memo: claims before the merge, copies after (counted with k_misses)
    CK(cudaMemsetAsync(w.memo, 0xFF, w.memo_slots * sizeof(uint64_t), st));
    k_memo_claim<<<(unsigned)(8 * h->n_sms), kMemoThreads, 0, st>>>(d_bytes, w.misses, w.miss_cap, w.memo,
                                                                    w.memo_slots - 1, w.follow, h->d_small);
    CK(cudaGetLastError());
  }
  k_misses<<<(unsigned)(kMissBlocksPerSm * h->n_sms), kMissThreads, 0, st>>>(d_bytes, w.misses, w.miss_cap, w.follow,
                                                                            w.stage, w.rec, a.T, h->d_small);
  if (w.memo) {
    CK(cudaGetLastError());
    k_memo_copy<<<(unsigned)(8 * h->n_sms), kMemoThreads, 0, st>>>(w.misses, w.miss_cap, w.follow, w.stage, w.rec,
                                                                   h->d_small);
  }
  CK(cudaGetLastError());
  if (ev_phase) CK(cudaEventRecord(ev_phase[phase++], st));
  k_giants<<<(unsigned)(8 * h->n_sms), kGiantThreads, 0, st>>>(d_bytes, w.giants, w.giant_cap, w.first_start, n_tiles,
                                                            w.rec, w.pool, a.T, h->d_small);
  CK(cudaGetLastError());
  if (ev_phase) CK(cudaEventRecord(ev_phase[phase++], st));
  const int64_t n_blocks = (n_tiles + kScanThreads - 1) / kScanThreads;
  k_scan_tiles<<<(unsigned)n_blocks, kScanThreads, 0, st>>>(w.rec, n_tiles, w.tile_base, w.block_sum);
  CK(cudaGetLastError());
  if (ev_phase) CK(cudaEventRecord(ev_phase[phase++], st));
  k_scan_tile_sums<<<1, kScanThreads, 0, st>>>(w.block_sum, n_blocks, h->d_small);
  CK(cudaGetLastError());
  if (ev_phase) CK(cudaEventRecord(ev_phase[phase++], st));
  k_compact<<<(unsigned)std::min<int64_t>((n_tiles + kCompactWarps - 1) / kCompactWarps, 8 * h->n_sms),
              32 * kCompactWarps, 0, st>>>(w.rec, w.stage, w.tile_base, w.block_sum, w.giants, w.giant_cap,
                                          d_doc_offsets, n_tiles, d_out_ids, out_capacity, d_out_offsets, h->d_small);
  CK(cudaGetLastError());
  if (ev_phase) CK(cudaEventRecord(ev_phase[phase++], st));
  k_giant_copy<<<(unsigned)(4 * h->n_sms), kCopyThreads, 0, st>>>(w.giants, w.giant_cap, w.pool, d_out_ids,
                                                                  out_capacity, h->d_small);
  CK(cudaGetLastError());
  if (ev_phase) CK(cudaEventRecord(ev_phase[phase++], st));
  if (ev_stop) CK(cudaEventRecord(ev_stop, st));
  static_assert(BPE_ENCODE_LAUNCHES == 9, "the launches above");
  return BPE_OK;
}
}  // namespace

extern "C" {

const char* bpe_last_error(void) { return g_err.c_str(); }

int bpe_build(const int32_t* merges, int64_t n_merges, const uint8_t* vocab_bytes, const int64_t* vocab_offsets,
              int64_t n_vocab, int device, bpe_handle** out) {
  if (!out || !vocab_offsets || (n_merges > 0 && !merges) || n_merges < 0 || n_vocab < 256)
    return fail(BPE_ERR_INVALID_ARG, "bpe_build: bad arguments");
  *out = nullptr;
  if (n_vocab > (1 << 20)) return fail(BPE_ERR_BAD_TABLE, "n_vocab above 2^20");
  if (n_merges >= (1 << 20) - 1) return fail(BPE_ERR_BAD_TABLE, "n_merges above 2^20 - 2");
  if (vocab_offsets[0] != 0) return fail(BPE_ERR_BAD_TABLE, "vocab_offsets[0] != 0");
  for (int64_t k = 0; k < n_vocab; ++k)
    if (vocab_offsets[k + 1] < vocab_offsets[k]) return fail(BPE_ERR_BAD_TABLE, "vocab_offsets not monotone");
  if (vocab_offsets[n_vocab] > 0 && !vocab_bytes) return fail(BPE_ERR_INVALID_ARG, "vocab_bytes is null");
  auto tok = [&](int64_t id) {
    return std::string((const char*)vocab_bytes + vocab_offsets[id], (size_t)(vocab_offsets[id + 1] - vocab_offsets[id]));
  };
  std::vector<int32_t> byte_id(256, -1);
  {
    std::unordered_set<std::string> seen;
    for (int64_t id = 0; id < n_vocab; ++id) {
      int64_t L = vocab_offsets[id + 1] - vocab_offsets[id];
      if (L == 0) continue;
      std::string s = tok(id);
      if (!seen.insert(s).second) return fail(BPE_ERR_BAD_TABLE, "two tokens have the same bytes");
      if (L == 1) byte_id[(uint8_t)s[0]] = (int32_t)id;
    }
    for (int b = 0; b < 256; ++b)
      if (byte_id[b] < 0) return fail(BPE_ERR_BAD_TABLE, "a single byte is missing from the vocabulary");
  }
  uint64_t nb = 1;
  while (nb < (uint64_t)n_merges) nb <<= 1;  // at most one entry per 2-slot bucket on average
  std::vector<uint4> ht(nb * 2, make_uint4(kEmptySlot, kEmptySlot, kInf, 0));
  {
    std::unordered_set<uint64_t> pairs;
    for (int64_t r = 0; r < n_merges; ++r) {
      int32_t a = merges[3 * r], b = merges[3 * r + 1], nw = merges[3 * r + 2];
      if (a < 0 || b < 0 || nw < 0 || a >= n_vocab || b >= n_vocab || nw >= n_vocab)
        return fail(BPE_ERR_BAD_TABLE, "merge id out of range");
      if (vocab_offsets[a + 1] == vocab_offsets[a] || vocab_offsets[b + 1] == vocab_offsets[b])
        return fail(BPE_ERR_BAD_TABLE, "merge uses an unused id");
      if (tok(nw) != tok(a) + tok(b)) return fail(BPE_ERR_BAD_TABLE, "bytes(new) != bytes(left) + bytes(right)");
      uint64_t key = ((uint64_t)(uint32_t)a << 20) | (uint32_t)b;
      if (!pairs.insert(key).second) return fail(BPE_ERR_BAD_TABLE, "a pair appears twice");
      uint64_t bucket = pair_hash((uint32_t)a, (uint32_t)b) & (nb - 1);
      for (;;) {
        int slot = -1;
        for (int q = 0; q < 2; ++q)
          if (ht[bucket * 2 + q].x == kEmptySlot) {
            slot = q;
            break;
          }
        if (slot >= 0) {
          ht[bucket * 2 + slot] = make_uint4((uint32_t)a, (uint32_t)b, (uint32_t)r, (uint32_t)nw);
          break;
        }
        bucket = (bucket + 1) & (nb - 1);
      }
    }
  }
  int n_dev = 0;
  CK(cudaGetDeviceCount(&n_dev));
  if (device < 0 || device >= n_dev) return fail(BPE_ERR_INVALID_ARG, "bad device ordinal");
  DeviceGuard g(device);
  bpe_handle* h = new bpe_handle();
  h->device = device;
  h->n_merges = n_merges;
  h->n_vocab = n_vocab;
  bpe_merges_monotone(merges, n_merges, n_vocab, &h->monotone);
  h->hmask = (uint32_t)(nb - 1);
  auto cleanup = [&](int code) {
    bpe_destroy(h);
    return code;
  };
#define CKB(call)                                                \
  do {                                                           \
    cudaError_t e_ = (call);                                     \
    if (e_ != cudaSuccess) return cleanup(cuda_fail(e_, #call)); \
  } while (0)
  CKB(cudaDeviceGetAttribute(&h->n_sms, cudaDevAttrMultiProcessorCount, device));
  CKB(cudaMalloc(&h->d_ht, ht.size() * sizeof(uint4)));
  CKB(cudaMemcpy(h->d_ht, ht.data(), ht.size() * sizeof(uint4), cudaMemcpyHostToDevice));
  CKB(cudaMalloc(&h->d_mrows, (size_t)std::max<int64_t>(1, n_merges) * 3 * sizeof(int32_t)));
  if (n_merges) CKB(cudaMemcpy(h->d_mrows, merges, (size_t)n_merges * 3 * sizeof(int32_t), cudaMemcpyHostToDevice));
  CKB(cudaMalloc(&h->d_byte_id, 256 * sizeof(int32_t)));
  CKB(cudaMemcpy(h->d_byte_id, byte_id.data(), 256 * sizeof(int32_t), cudaMemcpyHostToDevice));
  const int64_t nvb = vocab_offsets[n_vocab];
  CKB(cudaMalloc(&h->d_vbytes, (size_t)std::max<int64_t>(1, nvb)));
  if (nvb) CKB(cudaMemcpy(h->d_vbytes, vocab_bytes, (size_t)nvb, cudaMemcpyHostToDevice));
  CKB(cudaMalloc(&h->d_voffs, (size_t)(n_vocab + 1) * sizeof(int64_t)));
  CKB(cudaMemcpy(h->d_voffs, vocab_offsets, (size_t)(n_vocab + 1) * sizeof(int64_t), cudaMemcpyHostToDevice));
  {
    std::vector<uint4> vent((size_t)n_vocab, make_uint4(0, 0, 0, 0));
    for (int64_t id = 0; id < n_vocab; ++id) {
      const int64_t b0 = vocab_offsets[id], L = vocab_offsets[id + 1] - b0;
      uint32_t w[3] = {0, 0, 0};
      for (int64_t q = 0; q < L && q < (int64_t)kDecInline; ++q) w[q >> 2] |= (uint32_t)vocab_bytes[b0 + q] << (8 * (q & 3));
      vent[(size_t)id] = make_uint4(w[0], w[1], w[2], (uint32_t)L);
    }
    CKB(cudaMalloc(&h->d_vent, vent.size() * sizeof(uint4)));
    CKB(cudaMemcpy(h->d_vent, vent.data(), vent.size() * sizeof(uint4), cudaMemcpyHostToDevice));
  }
  CKB(cudaMalloc(&h->d_small, sizeof(DevSmall)));
  CKB(cudaMemset(h->d_small, 0, sizeof(DevSmall)));
  CKB(cudaMallocHost(&h->h_small, sizeof(DevSmall)));
#undef CKB
  int rc = build_word_cache(h, vocab_bytes, vocab_offsets, n_vocab);
  if (rc) return cleanup(rc);
  *out = h;
  return BPE_OK;
}

int bpe_destroy(bpe_handle* h) {
  if (!h) return fail(BPE_ERR_INVALID_ARG, "null handle");
  DeviceGuard g(h->device);
  cudaDeviceSynchronize();
  cudaFree(h->d_ht);
  cudaFree(h->d_mrows);
  cudaFree(h->d_byte_id);
  cudaFree(h->d_vbytes);
  cudaFree(h->d_voffs);
  cudaFree(h->d_vent);
  cudaFree(h->d_cache);
  cudaFree(h->d_small);
  cudaFree(h->d_ws);
  for (auto& sl : h->slot) {
    cudaFree(sl.bytes);
    cudaFree(sl.offs);
    cudaFree(sl.ids);
    cudaFree(sl.out_offs);
    if (sl.in) cudaEventDestroy(sl.in);
    if (sl.done) cudaEventDestroy(sl.done);
    if (sl.free) cudaEventDestroy(sl.free);
  }
  if (h->s_h2d) cudaStreamDestroy(h->s_h2d);
  if (h->s_d2h) cudaStreamDestroy(h->s_d2h);
  if (h->h_totals) cudaFreeHost(h->h_totals);
  if (h->h_small) cudaFreeHost(h->h_small);
  delete h;
  return BPE_OK;
}

int bpe_set_word_cache(bpe_handle* h, int enable) {
  if (!h) return fail(BPE_ERR_INVALID_ARG, "null handle");
  h->cache_enabled = enable ? 1 : 0;
  return BPE_OK;
}

int bpe_set_call_memo(bpe_handle* h, int mode) {
  if (!h || (mode != BPE_MEMO_OFF && mode != BPE_MEMO_ON && mode != BPE_MEMO_AUTO))
    return fail(BPE_ERR_INVALID_ARG, "bpe_set_call_memo: mode must be BPE_MEMO_OFF, BPE_MEMO_ON or BPE_MEMO_AUTO");
  h->call_memo = mode;
  return BPE_OK;
}

int bpe_set_timing_events(bpe_handle* h, void* ev_start, void* ev_stop) {
  if (!h) return fail(BPE_ERR_INVALID_ARG, "null handle");
  h->ev_start = (cudaEvent_t)ev_start;
  h->ev_stop = (cudaEvent_t)ev_stop;
  return BPE_OK;
}

int bpe_set_phase_events(bpe_handle* h, void** events, int n) {
  if (!h || (n != 0 && (n != BPE_ENCODE_LAUNCHES + 1 || !events)))
    return fail(BPE_ERR_INVALID_ARG, "bpe_set_phase_events: n must be 0 or BPE_ENCODE_LAUNCHES + 1");
  h->ev_phase = n ? reinterpret_cast<cudaEvent_t*>(events) : nullptr;
  return BPE_OK;
}

int bpe_table_info(const bpe_handle* h, int64_t* n_merges, int64_t* n_vocab) {
  if (!h) return fail(BPE_ERR_INVALID_ARG, "null handle");
  if (n_merges) *n_merges = h->n_merges;
  if (n_vocab) *n_vocab = h->n_vocab;
  return BPE_OK;
}

int bpe_workspace_bytes(const bpe_handle* h, int64_t* bytes) {
  if (!h || !bytes) return fail(BPE_ERR_INVALID_ARG, "bpe_workspace_bytes: bad arguments");
  *bytes = (int64_t)h->ws_bytes;
  return BPE_OK;
}

int bpe_table_monotone(const bpe_handle* h, int* monotone) {
  if (!h || !monotone) return fail(BPE_ERR_INVALID_ARG, "bpe_table_monotone: bad arguments");
  *monotone = h->monotone;
  return BPE_OK;
}

int bpe_merges_monotone(const int32_t* merges, int64_t n_merges, int64_t n_vocab, int* monotone) {
  if (!monotone || n_merges < 0 || n_vocab < 0 || (n_merges > 0 && !merges))
    return fail(BPE_ERR_INVALID_ARG, "bpe_merges_monotone: bad arguments");
  // made[id]: the lowest rank whose merge makes id (-1: a single byte or an
  // id no merge makes, which counts as present from the start)
  std::vector<int64_t> made((size_t)n_vocab, -1);
  for (int64_t r = n_merges - 1; r >= 0; --r) {
    const int32_t nw = merges[3 * r + 2];
    if (nw < 0 || nw >= n_vocab) return fail(BPE_ERR_BAD_TABLE, "bpe_merges_monotone: merge id out of range");
    made[(size_t)nw] = r;
  }
  int ok = 1;
  for (int64_t r = 0; r < n_merges && ok; ++r) {
    for (int q = 0; q < 2; ++q) {
      const int32_t id = merges[3 * r + q];
      if (id < 0 || id >= n_vocab) return fail(BPE_ERR_BAD_TABLE, "bpe_merges_monotone: merge id out of range");
      if (made[(size_t)id] >= r) ok = 0;
    }
  }
  *monotone = ok;
  return BPE_OK;
}

int bpe_sync_status(bpe_handle* h, bpe_stream_t stream) {
  if (!h) return fail(BPE_ERR_INVALID_ARG, "null handle");
  DeviceGuard g(h->device);
  DevSmall s;
  int rc = read_status(h, (cudaStream_t)stream, &s);
  if (rc) return rc;
  return status_code(s.status);
}

int bpe_encode_batch(bpe_handle* h, const uint8_t* d_bytes, int64_t n_bytes, const int64_t* d_doc_offsets,
                     int64_t n_docs, int32_t* d_out_ids, int64_t out_capacity, int64_t* d_out_offsets,
                     int64_t* h_total_tokens, bpe_stream_t stream) {
  if (!h || !d_doc_offsets || !d_out_offsets || n_bytes < 0 || n_docs < 0 || (n_bytes > 0 && !d_bytes))
    return fail(BPE_ERR_INVALID_ARG, "bpe_encode_batch: bad arguments");
  if (out_capacity < 0 || (out_capacity > 0 && !d_out_ids))
    return fail(BPE_ERR_INVALID_ARG, "bpe_encode_batch: bad output buffer");
  if ((reinterpret_cast<uintptr_t>(d_doc_offsets) & 7u) || (reinterpret_cast<uintptr_t>(d_out_offsets) & 7u) ||
      (reinterpret_cast<uintptr_t>(d_out_ids) & 3u))
    return fail(BPE_ERR_INVALID_ARG, "bpe_encode_batch: offsets must be 8-byte and ids 4-byte aligned");
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  // the per-call memo: on request, or (by default) when the word cache is off
  // and the misses are every pre-token; queue indices must fit in 32 bits
  const bool memo = (h->call_memo == BPE_MEMO_ON || (h->call_memo == BPE_MEMO_AUTO && !h->cache_enabled)) &&
                    ws_sizes(n_bytes).miss_cap < (int64_t)UINT32_MAX;
  int rc = ensure_ws(h, ws_sizes(n_bytes, memo).total);
  if (rc) return rc;
  if (!h->smem_set) {
    if ((rc = tiles_smem_setup())) return rc;
    h->smem_set = true;
  }
  rc = launch_encode(h, ws_carve(static_cast<unsigned char*>(h->d_ws), n_bytes, memo), d_bytes, n_bytes,
                     d_doc_offsets, n_docs, d_out_ids, out_capacity, d_out_offsets, st, h->ev_start, h->ev_stop,
                     h->ev_phase);
  if (rc) return rc;
  if (h_total_tokens) {
    DevSmall s;
    rc = read_status(h, st, &s);
    if (rc) return rc;
    *h_total_tokens = s.total;
    return status_code(s.status);
  }
  return BPE_OK;
}

int bpe_encode_batch_noalloc(bpe_handle* h, const uint8_t* d_bytes, int64_t n_bytes, const int64_t* d_doc_offsets,
                             int64_t n_docs, int32_t* d_out_ids, int64_t out_capacity, int64_t* d_out_offsets,
                             int64_t* h_total_tokens, bpe_stream_t stream) {
  if (!h || !d_doc_offsets || !d_out_offsets || n_bytes < 0 || n_docs < 0 || (n_bytes > 0 && !d_bytes))
    return fail(BPE_ERR_INVALID_ARG, "bpe_encode_batch_noalloc: bad arguments");
  if (out_capacity < 0 || (out_capacity > 0 && !d_out_ids))
    return fail(BPE_ERR_INVALID_ARG, "bpe_encode_batch_noalloc: bad output buffer");
  if ((reinterpret_cast<uintptr_t>(d_doc_offsets) & 7u) || (reinterpret_cast<uintptr_t>(d_out_offsets) & 7u) ||
      (reinterpret_cast<uintptr_t>(d_out_ids) & 3u))
    return fail(BPE_ERR_INVALID_ARG, "bpe_encode_batch_noalloc: offsets must be 8-byte and ids 4-byte aligned");
  if (n_bytes > kNoAllocMaxBytes)
    return fail(BPE_ERR_INVALID_ARG, "bpe_encode_batch_noalloc: n_bytes = " + std::to_string(n_bytes) +
                                         " is above its fixed scratch limit of " + std::to_string(kNoAllocMaxBytes) +
                                         " bytes (4 MiB); encode larger batches with bpe_encode_batch");
  DeviceGuard g(h->device);
  unsigned char* base = nullptr;
  int rc = noalloc_setup(h->device, &base);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  rc = launch_encode(h, ws_carve(base, n_bytes), d_bytes, n_bytes, d_doc_offsets, n_docs, d_out_ids, out_capacity,
                     d_out_offsets, st, nullptr, nullptr, nullptr);
  if (rc) return rc;
  if (h_total_tokens) {
    DevSmall s;
    rc = read_status(h, st, &s);
    if (rc) return rc;
    *h_total_tokens = s.total;
    return status_code(s.status);
  }
  return BPE_OK;
}

int bpe_encode_batch_host(bpe_handle* h, const uint8_t* h_bytes, int64_t n_bytes, const int64_t* h_doc_offsets,
                          int64_t n_docs, int32_t* h_out_ids, int64_t out_capacity, int64_t* h_out_offsets,
                          int64_t* h_total_tokens, bpe_stream_t stream) {
  if (!h || !h_doc_offsets || !h_out_offsets || n_bytes < 0 || n_docs < 0 || (n_bytes > 0 && !h_bytes))
    return fail(BPE_ERR_INVALID_ARG, "bpe_encode_batch_host: bad arguments");
  if (out_capacity < 0 || (out_capacity > 0 && !h_out_ids))
    return fail(BPE_ERR_INVALID_ARG, "bpe_encode_batch_host: bad output buffer");
  const int64_t b_first = h_doc_offsets[0], b_last = h_doc_offsets[n_docs];
  if (b_first < 0 || b_last < b_first || b_last > n_bytes)
    return fail(BPE_ERR_BAD_INPUT, "bpe_encode_batch_host: first or last document offset outside the buffer");
  DeviceGuard g(h->device);
  cudaStream_t cs = (cudaStream_t)stream;
  // Slices of whole documents, about T = (b_last - b_first) / 12 bytes each.
  // The first three ramp up (T/8, T/4, T/2) and the last ones halve down to
  // T/8, so the first encode starts, and the last download ends, soon after
  // the copies begin and end. No slice is asked for less than 4 MiB; a
  // document longer than its slice is a slice of its own.
  const int64_t T = std::max<int64_t>(int64_t(4) << 20, (b_last - b_first + 11) / 12);
  std::vector<int64_t> cut{0};
  while (cut.back() < n_docs) {
    const int64_t j = (int64_t)cut.size() - 1, d0 = cut.back(), rest = b_last - h_doc_offsets[d0];
    int64_t target = j < 3 ? T >> (3 - j) : (rest > 2 * T ? T : (rest > T / 4 ? rest / 2 : rest));
    target = std::max<int64_t>(target, int64_t(4) << 20);
    const int64_t want = h_doc_offsets[d0] + target;
    int64_t lo = d0 + 1, hi = n_docs;  // last doc boundary at or below want, at least one document
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) / 2;
      if (h_doc_offsets[mid] <= want) lo = mid;
      else hi = mid - 1;
    }
    const int64_t a = h_doc_offsets[d0], b = h_doc_offsets[lo];
    if (b < a || b > b_last) return fail(BPE_ERR_BAD_INPUT, "bpe_encode_batch_host: offsets not monotone");
    cut.push_back(lo);
  }
  const int64_t n_slices = std::max<int64_t>(1, (int64_t)cut.size() - 1);
  if (cut.size() == 1) cut.push_back(0);  // no documents: one empty slice
  int64_t max_bytes = 0, max_docs = 0;
  for (int64_t j = 0; j < n_slices; ++j) {
    max_bytes = std::max(max_bytes, h_doc_offsets[cut[j + 1]] - h_doc_offsets[cut[j]]);
    max_docs = std::max(max_docs, cut[j + 1] - cut[j]);
  }
  // Buffers, streams and events, grown or made on first need.
  if (max_bytes > h->slot_bytes || max_docs > h->slot_docs) {
    CK(cudaDeviceSynchronize());
    const int64_t nb = std::max(max_bytes, h->slot_bytes), nd = std::max(max_docs, h->slot_docs);
    for (auto& sl : h->slot) {
      cudaFree(sl.bytes);
      cudaFree(sl.offs);
      cudaFree(sl.ids);
      cudaFree(sl.out_offs);
      sl.bytes = nullptr;
      sl.offs = sl.out_offs = nullptr;
      sl.ids = nullptr;
    }
    h->slot_bytes = h->slot_docs = 0;
    for (auto& sl : h->slot) {
      CK(cudaMalloc(&sl.bytes, (size_t)std::max<int64_t>(16, nb)));
      CK(cudaMalloc(&sl.offs, (size_t)(nd + 1) * sizeof(int64_t)));
      CK(cudaMalloc(&sl.ids, (size_t)std::max<int64_t>(1, nb) * sizeof(int32_t)));
      CK(cudaMalloc(&sl.out_offs, (size_t)(nd + 1) * sizeof(int64_t)));
    }
    h->slot_bytes = nb;
    h->slot_docs = nd;
  }
  for (auto& sl : h->slot) {
    if (!sl.in) CK(cudaEventCreateWithFlags(&sl.in, cudaEventDisableTiming));
    if (!sl.done) CK(cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming));
    if (!sl.free) CK(cudaEventCreateWithFlags(&sl.free, cudaEventDisableTiming));
  }
  if (!h->s_h2d) CK(cudaStreamCreateWithFlags(&h->s_h2d, cudaStreamNonBlocking));
  if (!h->s_d2h) CK(cudaStreamCreateWithFlags(&h->s_d2h, cudaStreamNonBlocking));
  if (n_slices > h->h_totals_cap) {
    if (h->h_totals) CK(cudaFreeHost(h->h_totals));
    h->h_totals = nullptr;
    h->h_totals_cap = 0;
    CK(cudaMallocHost(&h->h_totals, (size_t)n_slices * sizeof(int64_t)));
    CK(cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->d_totals), h->h_totals, 0));
    h->h_totals_cap = n_slices;
  }
  int rc = ensure_ws(h, ws_sizes(h->slot_bytes).total);
  if (rc) return rc;
  if (!h->smem_set) {
    if ((rc = tiles_smem_setup())) return rc;
    h->smem_set = true;
  }
  // Slice j: upload (stream h2d) -> encode (the caller's stream) -> count to
  // the host -> shift offsets, download (stream d2h). Slot j % kHostSlots is
  // reused by slice j + kHostSlots once slice j's download is done.
  constexpr int NS = bpe_handle::kHostSlots;
  auto issue_in = [&](int64_t j) -> int {
    auto& sl = h->slot[j % NS];
    const int64_t d0 = cut[j], nd = cut[j + 1] - d0, b0 = h_doc_offsets[d0], nb = h_doc_offsets[cut[j + 1]] - b0;
    if (j >= NS) CK(cudaStreamWaitEvent(h->s_h2d, sl.free, 0));
    if (nb > 0) CK(cudaMemcpyAsync(sl.bytes, h_bytes + b0, (size_t)nb, cudaMemcpyHostToDevice, h->s_h2d));
    CK(cudaMemcpyAsync(sl.offs, h_doc_offsets + d0, (size_t)(nd + 1) * sizeof(int64_t), cudaMemcpyHostToDevice,
                       h->s_h2d));
    CK(cudaEventRecord(sl.in, h->s_h2d));
    CK(cudaStreamWaitEvent(cs, sl.in, 0));
    k_offsets_shift<<<(unsigned)std::min<int64_t>(1024, nd / 256 + 1), 256, 0, cs>>>(sl.offs, nd + 1, -b0);
    CK(cudaGetLastError());
    int r = launch_encode(h, ws_carve(static_cast<unsigned char*>(h->d_ws), nb), sl.bytes, nb, sl.offs, nd, sl.ids,
                          nb, sl.out_offs, cs, nullptr, nullptr, nullptr);
    if (r) return r;
    k_total_to_host<<<1, 32, 0, cs>>>(h->d_small, h->d_totals + j);
    CK(cudaGetLastError());
    CK(cudaEventRecord(sl.done, cs));
    return BPE_OK;
  };
  for (int64_t j = 0; j < std::min<int64_t>(NS, n_slices); ++j)
    if ((rc = issue_in(j))) return rc;
  int64_t base = 0;
  for (int64_t j = 0; j < n_slices; ++j) {
    auto& sl = h->slot[j % NS];
    const int64_t d0 = cut[j], nd = cut[j + 1] - d0;
    CK(cudaEventSynchronize(sl.done));
    const int64_t tot = h->h_totals[j];
    CK(cudaStreamWaitEvent(h->s_d2h, sl.done, 0));
    k_offsets_shift<<<(unsigned)std::min<int64_t>(1024, nd / 256 + 1), 256, 0, h->s_d2h>>>(sl.out_offs, nd + 1, base);
    CK(cudaGetLastError());
    const int64_t fit = std::max<int64_t>(0, std::min(tot, out_capacity - base));
    if (fit > 0)
      CK(cudaMemcpyAsync(h_out_ids + base, sl.ids, (size_t)fit * sizeof(int32_t), cudaMemcpyDeviceToHost, h->s_d2h));
    const int64_t n_out = nd + (j == n_slices - 1 ? 1 : 0);  // the next slice writes its first offset
    if (n_out > 0)
      CK(cudaMemcpyAsync(h_out_offsets + d0, sl.out_offs, (size_t)n_out * sizeof(int64_t), cudaMemcpyDeviceToHost,
                         h->s_d2h));
    CK(cudaEventRecord(sl.free, h->s_d2h));
    base += tot;
    if (j + NS < n_slices && (rc = issue_in(j + NS))) return rc;
  }
  CK(cudaStreamSynchronize(h->s_d2h));
  DevSmall s;
  rc = read_status(h, cs, &s);
  if (rc) return rc;
  if (h_total_tokens) *h_total_tokens = base;
  if (s.status) return status_code(s.status);
  if (base > out_capacity) return fail(BPE_ERR_CAPACITY, "output capacity exceeded");
  return BPE_OK;
}

int bpe_pretokenize_batch(const uint8_t* d_bytes, int64_t n_bytes, const int64_t* d_doc_offsets, int64_t n_docs,
                          uint32_t* d_start_bits, bpe_stream_t stream) {
  if (!d_doc_offsets || n_bytes < 0 || n_docs < 0 || (n_bytes > 0 && (!d_bytes || !d_start_bits)))
    return fail(BPE_ERR_INVALID_ARG, "bpe_pretokenize_batch: bad arguments");
  if (n_bytes == 0) return BPE_OK;
  const int64_t n_tiles = n_bytes / kTileOwn + 1;
  k_split_tiles<<<(unsigned)((n_tiles + kSplitWarps - 1) / kSplitWarps), 32 * kSplitWarps, 0, (cudaStream_t)stream>>>(
      d_bytes, n_bytes, d_doc_offsets, n_docs, n_tiles, d_start_bits);
  CK(cudaGetLastError());
  return BPE_OK;
}

int bpe_decode_batch(bpe_handle* h, const int32_t* d_ids, int64_t n_ids, const int64_t* d_id_offsets, int64_t n_docs,
                     uint8_t* d_out_bytes, int64_t out_capacity, int64_t* d_out_byte_offsets, int64_t* h_total_bytes,
                     bpe_stream_t stream) {
  if (!h || !d_id_offsets || !d_out_byte_offsets || n_ids < 0 || n_docs < 0 || out_capacity < 0 ||
      (n_ids > 0 && !d_ids) || (out_capacity > 0 && !d_out_bytes))
    return fail(BPE_ERR_INVALID_ARG, "bpe_decode_batch: bad arguments");
  if ((reinterpret_cast<uintptr_t>(d_id_offsets) & 7u) || (reinterpret_cast<uintptr_t>(d_out_byte_offsets) & 7u) ||
      (reinterpret_cast<uintptr_t>(d_ids) & 3u))
    return fail(BPE_ERR_INVALID_ARG, "bpe_decode_batch: offsets must be 8-byte and ids 4-byte aligned");
  DeviceGuard g(h->device);
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t n_tiles = n_ids / kDecIds + 1;
  const int64_t n_blocks = (n_tiles + kDecScanThreads - 1) / kDecScanThreads;
  const size_t a1 = align256((size_t)n_tiles * sizeof(uint64_t)), a2 = align256((size_t)n_blocks * sizeof(uint64_t));
  int rc = ensure_ws(h, a1 + a2 + align256((size_t)n_tiles * sizeof(int64_t)));
  if (rc) return rc;
  uint64_t* tile_base = reinterpret_cast<uint64_t*>(h->d_ws);
  uint64_t* block_sum = reinterpret_cast<uint64_t*>(static_cast<unsigned char*>(h->d_ws) + a1);
  int64_t* first_doc = reinterpret_cast<int64_t*>(static_cast<unsigned char*>(h->d_ws) + a1 + a2);
  const unsigned tile_grid = (unsigned)std::min<int64_t>((n_tiles + kDecWarps - 1) / kDecWarps, 8 * h->n_sms);
  k_dec_count<<<tile_grid, 32 * kDecWarps, 0, st>>>(d_ids, n_ids, h->d_vent, h->n_vocab, n_tiles, tile_base,
                                                    h->d_small);
  k_dec_scan_tiles<<<(unsigned)n_blocks, kDecScanThreads, 0, st>>>(tile_base, n_tiles, block_sum);
  k_scan_tile_sums<<<1, kScanThreads, 0, st>>>(block_sum, n_blocks, h->d_small);
  const int64_t n_first = std::max<int64_t>(n_tiles, n_docs + 1);
  k_dec_first_doc<<<(unsigned)std::min<int64_t>(4096, (n_first + 255) / 256), 256, 0, st>>>(d_id_offsets, n_docs, n_ids,
                                                                                           n_tiles, first_doc,
                                                                                           h->d_small);
  // k_dec_write: one wave (three CTAs fit an SM: registers and shared memory)
  const unsigned write_grid = (unsigned)std::min<int64_t>((n_tiles + kDecWarps - 1) / kDecWarps, 3 * h->n_sms);
  k_dec_write<<<write_grid, 32 * kDecWarps, 0, st>>>(d_ids, n_ids, h->d_vent, h->d_vbytes, h->d_voffs, h->n_vocab,
                                                    tile_base, block_sum, first_doc, d_id_offsets, n_docs, n_tiles,
                                                    d_out_bytes, out_capacity, d_out_byte_offsets, h->d_small);
  CK(cudaGetLastError());
  if (h_total_bytes) {
    DevSmall s;
    rc = read_status(h, st, &s);
    if (rc) return rc;
    *h_total_bytes = s.total;
    if (s.status) return status_code(s.status);
    if (s.total > out_capacity) return fail(BPE_ERR_CAPACITY, "decoded bytes exceed out_capacity");
  }
  return BPE_OK;
}

int bpe_train(const uint8_t* word_bytes, const int64_t* word_offsets, const int64_t* word_counts, int64_t n_words,
              int64_t n_merges, int device, int32_t* merges_out, int64_t* n_made) {
  if (n_words < 0 || n_merges < 0 || !word_offsets || (n_words > 0 && !word_counts) || !n_made ||
      (n_merges > 0 && !merges_out) || (word_offsets[n_words] > 0 && !word_bytes) ||
      n_merges > (int64_t)(1 << 20) - 256)
    return fail(BPE_ERR_INVALID_ARG, "bpe_train: bad arguments");
  if (word_offsets[0] != 0) return fail(BPE_ERR_INVALID_ARG, "bpe_train: word_offsets[0] must be 0");
  int64_t n_pairs = 0;
  std::vector<int32_t> len((size_t)std::max<int64_t>(1, n_words));
  for (int64_t w = 0; w < n_words; ++w) {
    const int64_t L = word_offsets[w + 1] - word_offsets[w];
    if (L < 0 || L > INT32_MAX || word_counts[w] < 0)
      return fail(BPE_ERR_INVALID_ARG, "bpe_train: offsets must not decrease and counts must be >= 0");
    len[(size_t)w] = (int32_t)L;
    n_pairs += L > 1 ? L - 1 : 0;
  }
  *n_made = 0;
  if (n_words == 0 || n_merges == 0) return BPE_OK;
  DeviceGuard g(device);
  const int64_t n_sym = word_offsets[n_words];
  std::vector<int32_t> sym((size_t)std::max<int64_t>(1, n_sym));
  for (int64_t i = 0; i < n_sym; ++i) sym[(size_t)i] = word_bytes[i];  // byte b is symbol b
  uint64_t n_slots = 1024;
  while (n_slots < (uint64_t)n_pairs * 2) n_slots <<= 1;
  int n_sms = 1;
  CK(cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, device));
  const unsigned word_grid = (unsigned)std::min<int64_t>((n_words + kTrainThreads - 1) / kTrainThreads, 8 * n_sms);
  const unsigned slot_grid = (unsigned)std::min<uint64_t>((n_slots + kTrainThreads - 1) / kTrainThreads, 4 * n_sms);
  const unsigned repl_grid = std::max(word_grid, slot_grid);
  struct Dev {
    int32_t* sym = nullptr;
    int64_t* off = nullptr;
    int32_t* len = nullptr;
    int64_t* freq = nullptr;
    uint64_t* keys = nullptr;
    unsigned long long* counts = nullptr;
    uint32_t* occ = nullptr;
    unsigned long long* bc = nullptr;
    unsigned long long* bk = nullptr;
    TrainState* st = nullptr;
    int32_t* merges = nullptr;
    cudaStream_t s = nullptr;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    ~Dev() {
      if (exec) cudaGraphExecDestroy(exec);
      if (graph) cudaGraphDestroy(graph);
      if (s) cudaStreamDestroy(s);
      cudaFree(sym); cudaFree(off); cudaFree(len); cudaFree(freq); cudaFree(keys); cudaFree(counts); cudaFree(occ);
      cudaFree(bc); cudaFree(bk); cudaFree(st); cudaFree(merges);
    }
  } d;
  CK(cudaMalloc(&d.sym, sym.size() * sizeof(int32_t)));
  CK(cudaMalloc(&d.off, (size_t)n_words * sizeof(int64_t)));
  CK(cudaMalloc(&d.len, (size_t)n_words * sizeof(int32_t)));
  CK(cudaMalloc(&d.freq, (size_t)n_words * sizeof(int64_t)));
  CK(cudaMalloc(&d.keys, n_slots * sizeof(uint64_t)));
  CK(cudaMalloc(&d.counts, n_slots * sizeof(unsigned long long)));
  CK(cudaMalloc(&d.occ, n_slots * sizeof(uint32_t)));
  CK(cudaMalloc(&d.bc, slot_grid * sizeof(unsigned long long)));
  CK(cudaMalloc(&d.bk, slot_grid * sizeof(unsigned long long)));
  CK(cudaMalloc(&d.st, sizeof(TrainState)));
  CK(cudaMalloc(&d.merges, (size_t)n_merges * 3 * sizeof(int32_t)));
  CK(cudaStreamCreateWithFlags(&d.s, cudaStreamNonBlocking));
  CK(cudaMemcpyAsync(d.sym, sym.data(), sym.size() * sizeof(int32_t), cudaMemcpyHostToDevice, d.s));
  CK(cudaMemcpyAsync(d.off, word_offsets, (size_t)n_words * sizeof(int64_t), cudaMemcpyHostToDevice, d.s));
  CK(cudaMemcpyAsync(d.len, len.data(), (size_t)n_words * sizeof(int32_t), cudaMemcpyHostToDevice, d.s));
  CK(cudaMemcpyAsync(d.freq, word_counts, (size_t)n_words * sizeof(int64_t), cudaMemcpyHostToDevice, d.s));
  CK(cudaMemsetAsync(d.keys, 0xFF, n_slots * sizeof(uint64_t), d.s));
  CK(cudaMemsetAsync(d.counts, 0, n_slots * sizeof(unsigned long long), d.s));
  CK(cudaMemsetAsync(d.st, 0, sizeof(TrainState), d.s));
  // kSteps identical steps per graph launch
  constexpr int kSteps = 64;
  CK(cudaStreamBeginCapture(d.s, cudaStreamCaptureModeThreadLocal));
  for (int k = 0; k < kSteps; ++k) {
    k_train_count<<<word_grid, kTrainThreads, 0, d.s>>>(d.sym, d.off, d.len, d.freq, n_words, d.keys, d.counts,
                                                         n_slots - 1, d.occ, d.st);
    k_train_best<<<slot_grid, kTrainThreads, 0, d.s>>>(d.keys, d.counts, d.occ, d.bc, d.bk, d.st, d.merges,
                                                        n_merges);
    k_train_replace<<<repl_grid, kTrainThreads, 0, d.s>>>(d.sym, d.off, d.len, n_words, d.keys, d.counts, d.occ,
                                                           d.st);
  }
  CK(cudaStreamEndCapture(d.s, &d.graph));
  CK(cudaGraphInstantiate(&d.exec, d.graph, 0));
  TrainState hs{};
  for (int64_t done_steps = 0; done_steps < n_merges;) {
    // up to 16 graph launches between looks at the state
    for (int r = 0; r < 16 && done_steps < n_merges; ++r, done_steps += kSteps) CK(cudaGraphLaunch(d.exec, d.s));
    CK(cudaMemcpyAsync(&hs, d.st, sizeof(TrainState), cudaMemcpyDeviceToHost, d.s));
    CK(cudaStreamSynchronize(d.s));
    if (hs.done) break;
  }
  CK(cudaMemcpyAsync(&hs, d.st, sizeof(TrainState), cudaMemcpyDeviceToHost, d.s));
  CK(cudaStreamSynchronize(d.s));
  const int64_t made = std::min<int64_t>(hs.made, n_merges);
  if (made > 0)
    CK(cudaMemcpy(merges_out, d.merges, (size_t)made * 3 * sizeof(int32_t), cudaMemcpyDeviceToHost));
  *n_made = made;
  return BPE_OK;
}

}  // extern "C"
