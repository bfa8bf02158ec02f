// Warp-tile encoder: the split, byte -> symbol and the word cache in one pass
// over the input, one warp per tile; the cache misses merged GPU-wide after
// it; then the ids placed by a scan of the tiles' counts.
//
// Included once by bpe_kernels.cu after the shared helpers (window, split
// masks, word cache, lane-group and CTA merges); not a standalone header.
//
// The method is the one bpe_kernels.cu describes (glitch4techs, "Tokenization
// LLM", sections "Technical analysis", "Byte-level encoding", "BPE merge
// algorithm", "Vocabulary lookup"; tokenwerk, "Tokenisierung", section "Byte
// Pair Encoding schrittweise"). What follows is GPU organisation only:
//
//   * Tiles (k_tiles). Tile t owns the pre-tokens that start in input bytes
//     [2016 t, 2016 t + 2016). Its warp loads bytes [2016 t - 16, 2016 t +
//     2064) into shared memory (16 bytes of context on each side of the 2048
//     bytes it splits); lane l computes the start bits of bytes [32 l, 32 l +
//     32) and [1024 + 32 l, 1024 + 32 l + 32) of the tile, so lane 31's second
//     word covers a 32-byte margin where the tile's last pre-token normally
//     ends. The input is read once.
//   * Per pre-token, one lane: a word-cache probe for 2 to 16 bytes (a single
//     byte is its own token). The ids go to the tile's stage slot at reserved
//     positions: a hit reserves its id count, a miss its byte length (ids
//     never outnumber bytes), a pre-token longer than kShortMax bytes or
//     running past the margin one placeholder.
//   * Misses (k_misses, GPU-wide): a lane per miss of up to 8 bytes, groups
//     of 8, 16 or 32 lanes for longer ones; each writes its ids at its
//     reserved position, marks the rest of the reservation as holes and adds
//     their number to its tile's record.
//   * Long pre-tokens (k_giants): a CTA each, in a pool at their own bytes.
//   * Output: a two-level scan of the tiles' final counts (k_scan_tiles,
//     k_scan_tile_sums), then k_compact moves every tile's ids into place
//     without the holes, gives each placeholder its output position, and
//     writes the document offsets; k_giant_copy copies the long pre-tokens'
//     ids there. No kernel waits on another CTA.

namespace {

constexpr int kTileWords = 64;                     // 32-byte start-bit words a tile computes (two per lane)
constexpr int kTileOwn = 32 * (kTileWords - 1);    // 2016 bytes whose pre-tokens a tile owns
constexpr int kTileBits = 32 * kTileWords;         // 2048 bytes whose start bits a tile computes
using TileWin = WindowSmem<kTileBits, 0, true>;    // window: 16 + 2048 + 16 bytes
static_assert(TileWin::kLen == kHalo + kTileBits + kHalo, "tile window");
constexpr int kTileWarps = 8;                      // warps (tiles in flight) per CTA
constexpr int kTileThreads = 32 * kTileWarps;
constexpr int kTileCtasPerSm = 3;                  // resident CTAs (registers: at most 85 a thread)
constexpr int kMissCap = 128;                      // miss records a tile holds before it hands them on
constexpr int kMissFlush = kMissCap - 64;          // hand on once this many are held (a round adds <= 64)

// Span list entries (u16): the start's tile position, and flags.
constexpr uint32_t kSpanPos = 0x07FFu;
constexpr uint32_t kSpanNone = 0x07FFu;  // sentinel: no pre-token start in the margin
constexpr uint32_t kSpanSkip = 0x4000u;  // the end of the last document: nothing to encode
constexpr uint32_t kSpanDoc = 0x8000u;   // a document starts here

// Stage entries: an id (< 2^20), or a hole, or a placeholder for a deferred
// pre-token (its record index); kIdDoc marks the first id of a document.
constexpr uint32_t kIdDoc = 0x80000000u;
constexpr uint32_t kIdSpecial = 0x40000000u;
constexpr uint32_t kIdLong = 0x20000000u;
constexpr uint32_t kIdHole = kIdSpecial;
constexpr uint32_t kIdIndex = 0x1FFFFFFFu;

// A deferred pre-token (longer than kShortMax bytes, or running past its
// tile's margin): k_giants finds its end when unknown (-1), merges it into
// the pool at its own bytes and stores its id count; k_compact stores its
// output position, and k_giant_copy copies its ids there.
struct GiantRec {
  int64_t start;
  int64_t end;
  int64_t tile;
  int64_t at;
  uint32_t count;
  uint32_t pad;
};

// Per tile: its documents [k0, k1) (k = n_docs: the end of the last one),
// stage entries used, holes left by merged misses, extra ids of its
// deferred pre-tokens (their ids minus their placeholders), flags.
constexpr uint32_t kTileDup = 1u;   // two documents start at the same byte (an empty document)
struct TileRec {
  int64_t k0, k1;
  uint32_t resv;
  uint32_t holes;
  uint32_t extra;
  uint32_t flags;
};

// A tile's held miss record (u32): start | length << 11 | reserved position
// << 18 | document start << 29. Handed to k_misses as tile << 30 | the record.
constexpr int kMissLenShift = 11, kMissAtShift = 18, kMissDocShift = 29;
__device__ __forceinline__ uint64_t miss_entry(int64_t t, uint32_t rec) { return (uint64_t)t << 30 | rec; }

struct __align__(16) TileSmem {
  TileWin w;                      // the tile's window
  uint16_t span[kTileOwn + 8];    // pre-token starts
  uint32_t miss[kMissCap];        // held miss records
};
constexpr size_t kTileSmemBytes = 1024 + kTileWarps * sizeof(TileSmem);  // the CTA's byte map, then the warps
static_assert(kTileCtasPerSm * (kTileSmemBytes + 1024) <= 228 * 1024, "the tile CTAs fit in an SM's shared memory");

struct TileArgs {
  const uint8_t* bytes;
  int64_t n_bytes;
  const int64_t* doc_offsets;
  int64_t n_docs;
  Tables T;
  Cache C;
  const int64_t* first_doc;  // per tile: the first document starting at or after the window
  TileRec* rec;              // per tile
  int64_t* first_start;      // per tile: the first pre-token start it owns (INT64_MAX: none)
  uint32_t* stage;           // [n_tiles][kTileBits]
  uint64_t* misses;          // the miss queue
  int64_t miss_cap;
  GiantRec* giants;
  int64_t giant_cap;
  DevSmall* small;
  int64_t n_tiles;
};

__device__ __forceinline__ uint32_t lanemask_lt() {
  return (1u << (threadIdx.x & 31)) - 1u;
}

// Inclusive warp scan: each step adds the value d lanes below, using the
// valid-source predicate of shfl.sync.up instead of a lane comparison.
__device__ __forceinline__ uint32_t warp_scan_incl(uint32_t v) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    asm("{\n\t.reg .pred p;\n\t.reg .u32 r;\n\t"
        "shfl.sync.up.b32 r|p, %0, %1, 0, 0xffffffff;\n\t"
        "@p add.u32 %0, %0, r;\n\t}"
        : "+r"(v)
        : "r"(d));
  }
  return v;
}

// --------------------------------------------------------- window and docs --

// Bytes [t0 - kHalo, t0 + kTileBits + kHalo) into W.win (zero outside the
// input): 16-byte asynchronous copies when the input is 16-byte aligned
// (window offsets are multiples of 16), byte loads otherwise. The caller
// waits with cp_async_wait_all and __syncwarp.
__device__ void tile_load_bytes(TileWin& W, const uint8_t* bytes, int64_t n_bytes, int64_t t0, bool aligned) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = t0 - kHalo;
  if (aligned && w0 >= 0 && w0 + TileWin::kLen <= n_bytes) {  // the whole window exists (every tile but the edges)
    static_assert(TileWin::kLen == 130 * 16, "four copies per lane and two more");
    const uint8_t* g = bytes + w0 + 16 * lane;
#pragma unroll
    for (int c = 0; c < 4; ++c) cp_async16(W.win + 512 * c + 16 * lane, g + 512 * c);
    if (lane < 2) cp_async16(W.win + 2048 + 16 * lane, g + 2048);
    return;
  }
  for (int c = lane; c < TileWin::kLen / 16; c += 32) {
    const int64_t g = w0 + 16 * c;
    if (aligned && g >= 0 && g + 16 <= n_bytes) {
      cp_async16(W.win + 16 * c, bytes + g);
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) W.win[16 * c + k] = (g + k >= 0 && g + k < n_bytes) ? bytes[g + k] : 0;
    }
  }
}

struct TileDocs {
  int64_t k0, k1;  // documents starting in the tile's own bytes: [k0, k1)
  bool dup;        // two of them start at the same byte (an empty document)
};

// Document edges of the window into W.docbits (every offset, the end of the
// last document included) and the bytes outside every document into
// W.outbits; kA = the first document at or after the window start (clamped
// here). Offsets are read in warp-wide groups until one lies past the window
// or they stop increasing (malformed input: k_prep_docs reports it).
__device__ TileDocs tile_load_docs(TileWin& W, const int64_t* doc_offsets, int64_t n_docs, int64_t t0, int64_t kA,
                                   int64_t d_first, int64_t d_last) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = t0 - kHalo, w_end = w0 + TileWin::kLen;
  const bool inside = w0 >= d_first && w0 + 32 * (TileWin::kWords + 2) <= d_last;  // no byte outside the documents
  for (int i = lane; i < TileWin::kWords + 2; i += 32) {
    W.docbits[i] = 0;
    uint32_t word = 0;
    const int64_t p = w0 + 32 * i;
    if (!inside && (p < d_first || p + 32 > d_last)) {
      for (int k = 0; k < 32; ++k)
        if (p + k < d_first || p + k >= d_last) word |= 1u << k;
    }
    W.outbits[i] = word;
  }
  __syncwarp();
  kA = kA < 0 ? 0 : (kA > n_docs + 1 ? n_docs + 1 : kA);
  int64_t n_lt0 = 0, n_lt1 = 0, prev_last = INT64_MIN;
  bool dup = false;
  for (int64_t k = kA; k <= n_docs; k += 32) {
    const int64_t kk = k + lane;
    const int64_t o = kk <= n_docs ? __ldg(doc_offsets + kk) : INT64_MAX;
    if (o >= w0 && o < w_end) {
      const int i = (int)(o - w0);
      atomicOr(&W.docbits[i >> 5], 1u << (i & 31));
    }
    n_lt0 += __popc(__ballot_sync(0xFFFFFFFFu, o < t0));
    n_lt1 += __popc(__ballot_sync(0xFFFFFFFFu, o < t0 + kTileOwn));
    int64_t o_prev = __shfl_up_sync(0xFFFFFFFFu, o, 1);
    if (lane == 0) o_prev = prev_last;
    dup |= __any_sync(0xFFFFFFFFu, o == o_prev && o >= t0 && o < t0 + kTileOwn);
    const bool down = __any_sync(0xFFFFFFFFu, kk <= n_docs && o < o_prev);
    prev_last = __shfl_sync(0xFFFFFFFFu, o, 31);
    if (down || prev_last >= w_end) break;
  }
  __syncwarp();
  return TileDocs{kA + n_lt0, kA + n_lt1, dup};
}

// ------------------------------------------------------------- ASCII split --
// Start bits of window positions [p0, p0 + 32) (p0 a multiple of 16) when
// bytes p0 - 4 .. p0 + 35 are all ASCII; returns false otherwise (the caller
// then takes start_mask32, which handles every input). The rules are those of
// start_mask32 (B0..B3 of the split predicate) on 32-bit masks in byte order:
//   * per word, carry-free SWAR range tests give 0x80 in each byte that is a
//     letter, a digit, whitespace or U+0020;
//   * a multiply gathers those bits: for flag words a (bytes 0..3) and b
//     (bytes 4..7), ((a >> 4) | b) * 0x204081 has the eight flags in byte
//     order in bits 24..31 (each partial product lands on its own bit);
//   * B2 = S & (~prev S | (~next S & ~next doc start)), B3 = ~S & ~prev U+0020
//     & (prev S | class change among letter / digit / other), plus the
//     document starts, minus the bytes outside every document;
//   * each apostrophe at p0 - 3 .. p0 + 31 then resolves its contraction:
//     when it is eligible (a document start, or after a letter, a digit or
//     whitespace other than U+0020) and one of s t m d (or re ve ll) follows
//     in its document, the byte after it loses its start (B0) and the byte
//     after the suffix gets one (B1).
__device__ __forceinline__ uint4 lds_u128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"((unsigned)__cvta_generic_to_shared(p)));
  return v;
}

// Bits 24..31 of p0..p3 -> one word (p0's in byte 0).
__device__ __forceinline__ uint32_t gather32(uint32_t p0, uint32_t p1, uint32_t p2, uint32_t p3) {
  return __byte_perm(__byte_perm(p0, p1, 0x0073u), __byte_perm(p2, p3, 0x0073u), 0x5410u);
}

__device__ __forceinline__ bool ascii_letter(uint32_t b) { return (uint32_t)((b | 0x20u) - 'a') < 26u; }
__device__ __forceinline__ bool ascii_digit(uint32_t b) { return (uint32_t)(b - '0') < 10u; }
__device__ __forceinline__ bool ascii_space(uint32_t b) { return b == 0x20u || (uint32_t)(b - 9u) < 5u; }

template <class SS>
__device__ __forceinline__ bool ascii_split32(const SS& W, int p0, uint32_t* out) {
  const uint4 a = lds_u128(W.win + p0), b = lds_u128(W.win + p0 + 16);
  const uint32_t wp = lds_u32(reinterpret_cast<const uint32_t*>(W.win + p0) - 1);
  const uint32_t wn = lds_u32(reinterpret_cast<const uint32_t*>(W.win + p0 + 32));
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  if ((a.x | a.y | a.z | a.w | b.x | b.y | b.z | b.w | wp | wn) & 0x80808080u) return false;
  Flags4 f[8];
  uint32_t apos = 0;  // nonzero: an apostrophe among bytes p0 - 3 .. p0 + 31
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    f[m] = ascii_flags(w[m]);
    const uint32_t x = w[m] ^ 0x27272727u;
    apos |= (x - 0x01010101u) & ~x;
  }
  {
    const uint32_t x = (wp ^ 0x27272727u) | 0xFFu;  // bytes p0 - 3 .. p0 - 1
    apos |= (x - 0x01010101u) & ~x;
  }
  const uint32_t L = gather32(gather8(f[0].L, f[1].L), gather8(f[2].L, f[3].L), gather8(f[4].L, f[5].L),
                              gather8(f[6].L, f[7].L));
  const uint32_t N = gather32(gather8(f[0].N, f[1].N), gather8(f[2].N, f[3].N), gather8(f[4].N, f[5].N),
                              gather8(f[6].N, f[7].N));
  const uint32_t S = gather32(gather8(f[0].S, f[1].S), gather8(f[2].S, f[3].S), gather8(f[4].S, f[5].S),
                              gather8(f[6].S, f[7].S));
  const uint32_t SP = gather32(gather8(f[0].SP, f[1].SP), gather8(f[2].SP, f[3].SP), gather8(f[4].SP, f[5].SP),
                               gather8(f[6].SP, f[7].SP));
  // the byte before (p0 - 1) and after (p0 + 32)
  const uint32_t bp = wp >> 24, bn = wn & 0xFFu;
  const uint32_t pL = (L << 1) | (ascii_letter(bp) ? 1u : 0u), pN = (N << 1) | (ascii_digit(bp) ? 1u : 0u);
  const uint32_t pS = (S << 1) | (ascii_space(bp) ? 1u : 0u), pSP = (SP << 1) | (bp == 0x20u ? 1u : 0u);
  const uint32_t nS = (S >> 1) | (ascii_space(bn) ? 0x80000000u : 0u);
  const uint32_t D = bits32_at(W.docbits, p0), nD = bits32_at(W.docbits, p0 + 1);
  const uint32_t B2 = S & (~pS | (~nS & ~nD));
  const uint32_t B3 = ~S & ~pSP & (pS | (L ^ pL) | (N ^ pN));
  uint32_t base = B2 | B3 | D;
  if (apos & 0x80808080u) {
    // contractions, one apostrophe at a time: bit k of A is byte p0 - 3 + k
    uint32_t fa[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) fa[m] = ~((w[m] ^ 0x27272727u) + 0x7F7F7F7Fu) & 0x80808080u;
    const uint32_t own = gather32(gather8(fa[0], fa[1]), gather8(fa[2], fa[3]), gather8(fa[4], fa[5]),
                                  gather8(fa[6], fa[7]));
    const uint32_t before = movemask4(~((wp ^ 0x27272727u) + 0x7F7F7F7Fu) & 0x80808080u) >> 1;  // bytes p0-3..p0-1
    uint64_t A = ((uint64_t)own << 3) | before;
    while (A) {
      const int j = __ffsll((long long)A) - 1 - 3;
      A &= A - 1;
      const int q = p0 + j;
      const bool at_start = bit_at(W.docbits, q);
      const uint32_t c = W.win[q - 1];
      const bool eligible = at_start || ascii_letter(c) || ascii_digit(c) || (ascii_space(c) && c != 0x20u);
      if (!eligible || bit_at(W.docbits, q + 1)) continue;
      const uint32_t s1 = W.win[q + 1];
      int k = 0;
      if (s1 == 's' || s1 == 't' || s1 == 'm' || s1 == 'd') k = 1;
      else if (!bit_at(W.docbits, q + 2) && is_suffix2(s1, W.win[q + 2])) k = 2;
      if (!k) continue;
      if (j + 1 >= 0 && j + 1 < 32) base &= ~(1u << (j + 1));
      if (j + 1 + k >= 0 && j + 1 + k < 32) base |= 1u << (j + 1 + k);
    }
  }
  *out = base & ~bits32_at(W.outbits, p0);
  return true;
}

// A word-cache key from the window (tile positions [s, s + len), len <= 16).
__device__ __forceinline__ CacheKey tile_key(const TileWin& W, int s, int len) {
  const int ws = kHalo + s;
  const uint32_t* wv = reinterpret_cast<const uint32_t*>(W.win) + (ws >> 2);
  const uint32_t sh = (uint32_t)(ws & 3) * 8u;
  const uint32_t a0 = lds_u32(wv), a1 = lds_u32(wv + 1), a2 = lds_u32(wv + 2), a3 = lds_u32(wv + 3),
                 a4 = lds_u32(wv + 4);
  // word k keeps its low min(max(8 len - 32 k, 0), 32) bits: the top word of
  // (0 : ~0) shifted left by that many (the shift clamps at 32)
  const int nbit = 8 * len;
  CacheKey K;
  K.x0 = __funnelshift_r(a0, a1, sh) & __funnelshift_lc(~0u, 0u, (uint32_t)nbit);
  K.x1 = __funnelshift_r(a1, a2, sh) & __funnelshift_lc(~0u, 0u, (uint32_t)max(nbit - 32, 0));
  K.x2 = __funnelshift_r(a2, a3, sh) & __funnelshift_lc(~0u, 0u, (uint32_t)max(nbit - 64, 0));
  K.x3 = __funnelshift_r(a3, a4, sh) & __funnelshift_lc(~0u, 0u, (uint32_t)max(nbit - 96, 0));
  return K;
}

// The rest of a word-cache probe chain past the home slot: {count, id0, id1,
// id2} of key (x0..x3, len), count 0 when absent. The home slot settles
// almost every probe (the table is at most 1/16 full), so this is kept out of
// line, and takes and returns values only, so the caller's registers never
// need a memory address.
__device__ __noinline__ uint4 cache_probe_chain(const uint4* e, uint32_t mask, uint32_t x0, uint32_t x1, uint32_t x2,
                                                uint32_t x3, uint32_t len) {
  uint32_t slot = cache_hash(x0, x1, x2, x3, len) & mask;
  for (uint32_t probe = 0; probe < mask; ++probe) {
    slot = (slot + 1) & mask;
    uint4 ea, eb;
    ldg32(e + 2 * slot, ea, eb);
    if (eb.x == 0) break;
    if ((eb.x & 31u) == len && ea.x == x0 && ea.y == x1 && ea.z == x2 && ea.w == x3)
      return make_uint4((eb.x >> 5) & 7u, eb.y, eb.z, eb.w);
  }
  return make_uint4(0u, 0u, 0u, 0u);
}

// The held miss records of tile t into the GPU-wide queue (one atomic per
// hand-over).
__device__ void tile_hand_misses(const TileSmem& S, int n_miss, int64_t t, const TileArgs& a) {
  const int lane = threadIdx.x & 31;
  unsigned long long base = 0;
  if (lane == 0) base = atomicAdd(&a.small->n_misses, (unsigned long long)n_miss);
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  for (int i = lane; i < n_miss; i += 32) {
    if ((int64_t)(base + i) < a.miss_cap) a.misses[base + i] = miss_entry(t, S.miss[i]);
    else atomicOr(&a.small->status, kStInternal);
  }
}

// ---------------------------------------------------------------- kernel --

// Persistent: each warp takes tiles from a counter.
__global__ void __launch_bounds__(kTileThreads, kTileCtasPerSm) k_tiles(TileArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  int32_t* byte_id = reinterpret_cast<int32_t*>(smem_raw);
  TileSmem& S = reinterpret_cast<TileSmem*>(smem_raw + 1024)[threadIdx.x >> 5];
  TileWin& W = S.w;
  for (int i = threadIdx.x; i < 256; i += kTileThreads) byte_id[i] = a.T.byte_id[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const bool aligned = (reinterpret_cast<uintptr_t>(a.bytes) & 15u) == 0;
  int64_t d_first = __ldg(a.doc_offsets), d_last = __ldg(a.doc_offsets + a.n_docs);
  d_first = d_first < 0 ? 0 : (d_first > a.n_bytes ? a.n_bytes : d_first);
  d_last = d_last < d_first ? d_first : (d_last > a.n_bytes ? a.n_bytes : d_last);
  for (;;) {
    unsigned long long tu = 0;
    if (lane == 0) tu = atomicAdd(&a.small->tile_ctr, 1ull);
    const int64_t t = (int64_t)__shfl_sync(0xFFFFFFFFu, tu, 0);
    if (t >= a.n_tiles) break;
    const int64_t t0 = t * (int64_t)kTileOwn;
    tile_load_bytes(W, a.bytes, a.n_bytes, t0, aligned);
    const TileDocs D = tile_load_docs(W, a.doc_offsets, a.n_docs, t0, __ldg(a.first_doc + t), d_first, d_last);
    cp_async_wait_all();
    __syncwarp();

    // Split: lane l's two words of 32 start bits (tile bytes 32 l and 1024 +
    // 32 l); the end of the last document ends the pre-token before it.
    uint32_t m[2], dw[2], dso[2];
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
      const int p0 = kHalo + 1024 * hw + 32 * lane;
      dw[hw] = bits32_at(W.docbits, p0);
      dso[hw] = dw[hw] & bits32_at(W.outbits, p0);
      if (!ascii_split32(W, p0, &m[hw])) m[hw] = start_mask32(W, p0, false);  // a byte above 0x7F is near
      m[hw] |= dso[hw];
    }
    const bool own1 = lane < 31;  // lane 31's second word is the margin
    const uint32_t c0 = __popc(m[0]), c1 = own1 ? __popc(m[1]) : 0u;
    const uint32_t incl = warp_scan_incl(c0 | c1 << 16);
    const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t n_spans = (tot & 0xFFFFu) + (tot >> 16);
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
      if (hw == 1 && !own1) continue;
      uint32_t b = m[hw];
      uint32_t o = hw == 0 ? (incl & 0xFFFFu) - c0 : (tot & 0xFFFFu) + (incl >> 16) - c1;
      while (b) {
        const int k = __ffs(b) - 1;
        b &= b - 1;
        uint32_t v = (uint32_t)(1024 * hw + 32 * lane + k);
        if ((dw[hw] >> k) & 1u) v |= kSpanDoc;
        if ((dso[hw] >> k) & 1u) v |= kSpanSkip;
        S.span[o++] = (uint16_t)v;
      }
    }
    if (lane == 31) {
      S.span[n_spans] = (uint16_t)(m[1] ? (uint32_t)(kTileOwn + __ffs(m[1]) - 1) : kSpanNone);
      S.span[n_spans + 1] = (uint16_t)kSpanNone;
    }
    __syncwarp();
    if (lane == 0) a.first_start[t] = n_spans ? t0 + (int64_t)(S.span[0] & kSpanPos) : INT64_MAX;

    // Pre-tokens, two per lane per round: cache probes in flight together.
    uint32_t* stage = a.stage + t * (int64_t)kTileBits;
    uint32_t resv = 0;
    int n_miss = 0;
    enum : uint32_t { kNoPiece = 0, kProbe = 2, kMiss = 3, kLong = 4, kOne = 5 };
    for (uint32_t i0 = 0; i0 < n_spans; i0 += 64) {
      // Two slots per lane: i = i0 + lane and i0 + 32 + lane. Everything but
      // the rare cases is computed for every lane without branches (a slot
      // past the list reads the sentinel and is made no piece).
      uint32_t s[2], len[2], kind[2], doc[2];
      CacheKey K[2];
      uint4 ea[2], eb[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t i = i0 + 32u * h + lane;
        const uint32_t ic = min(i, n_spans);
        const uint32_t e0 = S.span[ic], e1 = S.span[ic + 1];
        s[h] = e0 & kSpanPos;
        len[h] = (e1 & kSpanPos) - s[h];
        doc[h] = (e0 & kSpanDoc) ? kIdDoc : 0u;
        const bool valid = i < n_spans && !(e0 & kSpanSkip);
        const bool lng = e1 == kSpanNone || len[h] > (uint32_t)kShortMax;
        kind[h] = !valid ? kNoPiece
                         : (lng ? kLong
                                : (len[h] == 1 ? kOne
                                               : ((len[h] <= (uint32_t)kCacheMaxLen && a.C.enabled) ? kProbe : kMiss)));
        K[h] = tile_key(W, (int)s[h], (int)min(len[h], (uint32_t)kCacheMaxLen));
        const uint32_t slot = cache_slot(K[h], len[h], a.C);
        ldg32(a.C.e + 2 * slot, ea[h], eb[h]);  // every lane: no branch (the slot is in range; unused unless probed)
      }
      uint32_t cnt[2], idv[2][kCacheMaxIds];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        // a probe's answer from its home slot, a single byte's id from the
        // byte map; the rest of a probe chain only when the home slot holds
        // another key
        const bool same = (eb[h].x & 31u) == len[h] &&
                          ((ea[h].x ^ K[h].x0) | (ea[h].y ^ K[h].x1) | (ea[h].z ^ K[h].x2) | (ea[h].w ^ K[h].x3)) == 0;
        const bool one = kind[h] == kOne;
        cnt[h] = one ? 1u : (same ? (eb[h].x >> 5) & 7u : 0u);
        idv[h][0] = one ? (uint32_t)byte_id[W.win[kHalo + s[h]]] : eb[h].y;
        idv[h][1] = eb[h].z;
        idv[h][2] = eb[h].w;
        if (kind[h] == kProbe && !same && eb[h].x != 0) {
          const uint4 r = cache_probe_chain(a.C.e, a.C.mask, K[h].x0, K[h].x1, K[h].x2, K[h].x3, len[h]);
          cnt[h] = r.x;
          idv[h][0] = r.y;
          idv[h][1] = r.z;
          idv[h][2] = r.w;
        }
        if (one || (kind[h] == kProbe && cnt[h])) kind[h] = kProbe;
        else if (kind[h] == kProbe) kind[h] = kMiss;
      }
      // reserved stage entries: a hit its ids, a miss its bytes, a long
      // pre-token one placeholder; both slots in one scan (16 bits each)
      const uint32_t r0 = kind[0] == kProbe ? cnt[0] : (kind[0] == kMiss ? len[0] : (kind[0] == kLong ? 1u : 0u));
      const uint32_t r1 = kind[1] == kProbe ? cnt[1] : (kind[1] == kMiss ? len[1] : (kind[1] == kLong ? 1u : 0u));
      const uint32_t incl = warp_scan_incl(r0 | r1 << 16);
      const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
      const uint32_t at[2] = {resv + (incl & 0xFFFFu) - r0, resv + (tot & 0xFFFFu) + (incl >> 16) - r1};
      resv += (tot & 0xFFFFu) + (tot >> 16);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (kind[h] == kProbe) {
          stage[at[h]] = idv[h][0] | doc[h];
          if (cnt[h] > 1) stage[at[h] + 1] = idv[h][1];
          if (cnt[h] > 2) stage[at[h] + 2] = idv[h][2];
        } else if (kind[h] == kLong) {
          const uint32_t end = (S.span[min(i0 + 32u * h + lane, n_spans) + 1] == kSpanNone) ? 0u : len[h];
          const unsigned long long gi = atomicAdd(&a.small->n_giants, 1ull);
          if ((int64_t)gi < a.giant_cap) {
            a.giants[gi] = GiantRec{t0 + (int64_t)s[h], end ? t0 + (int64_t)(s[h] + end) : -1, t, -1, 0u, 0u};
            stage[at[h]] = kIdSpecial | kIdLong | (uint32_t)gi | doc[h];
          } else {
            atomicOr(&a.small->status, kStInternal);
            stage[at[h]] = kIdHole;
          }
        }
        const bool miss = kind[h] == kMiss;
        const uint32_t mb = __ballot_sync(0xFFFFFFFFu, miss);
        if (miss)
          S.miss[n_miss + __popc(mb & lanemask_lt())] = s[h] | (len[h] << kMissLenShift) |
                                                         (at[h] << kMissAtShift) | (doc[h] ? 1u << kMissDocShift : 0u);
        n_miss += __popc(mb);
      }
      __syncwarp();
      if (n_miss >= kMissFlush) {
        tile_hand_misses(S, n_miss, t, a);
        n_miss = 0;
        __syncwarp();
      }
    }
    if (n_miss) tile_hand_misses(S, n_miss, t, a);
    if (lane == 0) a.rec[t] = TileRec{D.k0, D.k1, resv, 0u, 0u, D.dup ? kTileDup : 0u};
    __syncwarp();
  }
}

// ------------------------------------------------------------------ misses --

// One thread merges a pre-token of n <= 8 bytes: symbols, pair ranks and
// merged ids in its own column of shared memory (x[i * kMissThreads], so the
// threads of a warp use distinct banks). A step takes the lowest rank,
// replaces its occurrences left to right without overlap while compacting,
// and looks up again only the pairs next to a merged symbol, two at a time.
// The final ids go to out[0 .. count).
constexpr int kMissThreads = 256;
constexpr int kTinyMax = 8;
struct TinyScratch {
  uint32_t sy[kTinyMax * kMissThreads], rk[kTinyMax * kMissThreads], nw[kTinyMax * kMissThreads];
};

__device__ uint32_t merge_thread(TinyScratch& Z, const uint8_t* src, uint32_t n, const Tables& T,
                                 const int32_t* byte_id, uint32_t* out) {
  uint32_t* sy = Z.sy + threadIdx.x;
  uint32_t* rk = Z.rk + threadIdx.x;
  uint32_t* nw = Z.nw + threadIdx.x;
  for (uint32_t i = 0; i < n; ++i) sy[i * kMissThreads] = (uint32_t)byte_id[src[i]];
  uint32_t redo = n > 1 ? (1u << (n - 1)) - 1u : 0u;  // pairs to look up
  for (;;) {
    while (redo) {
      const uint32_t p1 = __ffs(redo) - 1;
      redo &= redo - 1;
      const uint32_t p2 = redo ? __ffs(redo) - 1 : kNone;
      redo &= redo - 1;
      uint32_t r1, w1, r2 = kInf, w2 = 0;
      lookup_pair2(T, sy[p1 * kMissThreads], sy[(p1 + 1) * kMissThreads], p2 != kNone ? sy[p2 * kMissThreads] : kNone,
                   p2 != kNone ? sy[(p2 + 1) * kMissThreads] : 0u, &r1, &w1, &r2, &w2);
      rk[p1 * kMissThreads] = r1;
      nw[p1 * kMissThreads] = w1;
      if (p2 != kNone) {
        rk[p2 * kMissThreads] = r2;
        nw[p2 * kMissThreads] = w2;
      }
    }
    uint32_t best = kInf;
    for (uint32_t i = 0; i + 1 < n; ++i) best = min(best, rk[i * kMissThreads]);
    if (best == kInf) break;
    uint32_t m = 0;
    for (uint32_t i = 0; i < n; ++m) {
      if (i + 1 < n && rk[i * kMissThreads] == best) {
        sy[m * kMissThreads] = nw[i * kMissThreads];
        redo |= (1u << m) | (m ? 1u << (m - 1) : 0u);  // the merged symbol's pairs
        i += 2;
      } else {
        sy[m * kMissThreads] = sy[i * kMissThreads];
        rk[m * kMissThreads] = rk[i * kMissThreads];
        nw[m * kMissThreads] = nw[i * kMissThreads];
        i += 1;
      }
    }
    n = m;
    redo &= n > 1 ? (1u << (n - 1)) - 1u : 0u;
  }
  for (uint32_t i = 0; i < n; ++i) out[i] = sy[i * kMissThreads];
  return n;
}

// The queued cache misses of every tile, a warp per 32 queue entries: up to
// 8 bytes a lane each (merge_thread); then, in rounds, groups of 8 lanes take
// the misses of 9 to 16 bytes, groups of 16 those of 17 to 32, and the whole
// warp each longer one (merge_group). Each writes its ids at its reserved
// stage position, holes over the rest of the reservation, the document mark
// on its first id, and adds its holes to its tile's record.
constexpr int kMissBlocksPerSm = 5;
__global__ void __launch_bounds__(kMissThreads, kMissBlocksPerSm) k_misses(const uint8_t* bytes, const uint64_t* queue,
                                                                           int64_t queue_cap, const uint32_t* follow,
                                                                           uint32_t* stage, TileRec* rec, Tables T,
                                                                           DevSmall* small) {
  __shared__ GroupScratch grp[kMissThreads / 32];
  __shared__ TinyScratch tiny;
  __shared__ int32_t byte_id[256];
  const unsigned long long n_raw = small->n_misses;
  const uint64_t n_q = n_raw < (unsigned long long)queue_cap ? n_raw : (unsigned long long)queue_cap;
  if (n_q == 0) return;
  for (int i = threadIdx.x; i < 256; i += kMissThreads) byte_id[i] = T.byte_id[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  GroupScratch& W = grp[threadIdx.x >> 5];
  const uint64_t warps = (uint64_t)gridDim.x * (kMissThreads / 32);
  for (uint64_t q0 = ((uint64_t)blockIdx.x * (kMissThreads / 32) + (threadIdx.x >> 5)) * 32; q0 < n_q; q0 += warps * 32) {
    // an entry another miss of the same bytes stands for (follow, the per-call
    // memo) is left to k_memo_copy
    const bool own = q0 + lane < n_q && (!follow || follow[q0 + lane] == (uint32_t)(q0 + lane));
    const uint64_t e = q0 + lane < n_q ? queue[q0 + lane] : 0ull;
    const uint32_t len = own ? (uint32_t)(e >> kMissLenShift) & 0x7Fu : 0u;  // 0: no entry
    // where a queue entry's bytes, ids and tile record are
    auto src_of = [&](uint64_t x) { return bytes + (int64_t)(x >> 30) * kTileOwn + (int64_t)(x & 0x7FFu); };
    auto out_of = [&](uint64_t x) {
      return stage + (int64_t)(x >> 30) * kTileBits + ((x >> kMissAtShift) & 0x7FFu);
    };
    auto finish = [&](uint64_t x, uint32_t n, uint32_t cnt, uint32_t* out) {
      for (uint32_t q = cnt; q < n; ++q) out[q] = kIdHole;
      if ((x >> kMissDocShift) & 1u) out[0] |= kIdDoc;
      if (n > cnt) atomicAdd(&rec[(int64_t)(x >> 30)].holes, n - cnt);
    };
    uint32_t m8 = __ballot_sync(0xFFFFFFFFu, len > 8u && len <= (uint32_t)kCacheMaxLen);
    uint32_t m16 = __ballot_sync(0xFFFFFFFFu, len > (uint32_t)kCacheMaxLen && len <= 32u);
    uint32_t m32 = __ballot_sync(0xFFFFFFFFu, len > 32u);
    // One round: group g of G lanes takes the g-th entry of *mask (none past
    // its end); the round's entries leave the mask.
    auto round = [&](uint32_t* mask, auto merge, int G) {
      const int g = lane / G;
      uint32_t mm = *mask;
      for (int x = 0; x < g; ++x) mm &= mm - 1u;
      const bool on = mm != 0;
      const int src = on ? __ffs(mm) - 1 : 0;
      for (int x = 0; x < 32 / G; ++x) *mask &= *mask - 1u;
      const uint64_t ge = __shfl_sync(0xFFFFFFFFu, e, src);
      const uint32_t n = on ? (uint32_t)(ge >> kMissLenShift) & 0x7Fu : 0u;
      uint32_t* out = out_of(ge);
      const uint32_t cnt = merge(src_of(ge), n, out);
      __syncwarp();
      if (on && (lane & (G - 1)) == 0) finish(ge, n, cnt, out);
    };
    if (len != 0 && len <= 8u) {  // up to 8 bytes: each lane its own
      uint32_t* out = out_of(e);
      const uint32_t cnt = merge_thread(tiny, src_of(e), len, T, byte_id, out);
      finish(e, len, cnt, out);
    }
    __syncwarp();
    while (m8)
      round(&m8, [&](const uint8_t* src, uint32_t n, uint32_t* out) { return merge_group<8>(W, src, n, T, byte_id, out); }, 8);
    while (m16)
      round(&m16, [&](const uint8_t* src, uint32_t n, uint32_t* out) { return merge_group<16>(W, src, n, T, byte_id, out); }, 16);
    while (m32)
      round(&m32, [&](const uint8_t* src, uint32_t n, uint32_t* out) { return merge_group<32>(W, src, n, T, byte_id, out); }, 32);
  }
}

// ------------------------------------------------------------- preparation --

// Per call, before k_tiles: counters reset, offsets validated, and
// first_doc[t] = the first document k with doc_offsets[k] >= 2016 t - 16
// (n_docs + 1 if none). Thread k writes the tiles whose window start lies in
// (doc_offsets[k - 1], doc_offsets[k]]: at most kPrepSpan of them, and a
// longer run goes to a list that k_prep_long fills.
constexpr int64_t kPrepSpan = 16;

struct PrepRange {
  int64_t k, t_lo, t_hi;
};

__device__ __forceinline__ int64_t floor_div(int64_t a, int64_t b) {
  const int64_t q = a / b;
  return (a % b != 0 && ((a < 0) != (b < 0))) ? q - 1 : q;
}

__global__ void k_prep_docs(const int64_t* doc_offsets, int64_t n_docs, int64_t n_bytes, int64_t n_tiles,
                            int64_t* first_doc, PrepRange* ranges, int64_t range_cap, DevSmall* small) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t0 == 0) {
    small->total = 0;
    small->tile_ctr = 0;
    small->n_misses = 0;
    small->n_giants = 0;
    small->giant_ctr = 0;
    // n_ranges is counted by this kernel's threads, so it starts the call at
    // zero from the call before (k_scan_tile_sums) or from bpe_build
  }
  bool bad = false;
  for (int64_t k = t0; k <= n_docs + 1; k += stride) {
    const int64_t prev = k == 0 ? INT64_MIN : __ldg(doc_offsets + k - 1);
    const int64_t cur = k <= n_docs ? __ldg(doc_offsets + k) : INT64_MAX;
    if (k <= n_docs && (cur < 0 || cur > n_bytes || (k > 0 && cur < prev))) {
      bad = true;
      continue;
    }
    int64_t lo = prev == INT64_MIN ? 0 : floor_div(prev + kHalo, kTileOwn) + 1;
    int64_t hi = cur == INT64_MAX ? n_tiles - 1 : floor_div(cur + kHalo, kTileOwn);
    lo = lo < 0 ? 0 : lo;
    hi = hi > n_tiles - 1 ? n_tiles - 1 : hi;
    if (hi - lo + 1 > kPrepSpan) {
      const unsigned long long i = atomicAdd(&small->n_ranges, 1ull);
      if ((int64_t)i < range_cap) ranges[i] = PrepRange{k, lo + kPrepSpan, hi};
      else bad = true;
      hi = lo + kPrepSpan - 1;
    }
    for (int64_t t = lo; t <= hi; ++t) first_doc[t] = k;
  }
  if (bad) atomicOr(&small->status, kStBadInput);
}

// The long runs of tiles k_prep_docs listed, a CTA per run; skipped when the
// offsets are malformed (the runs may then overlap without bound).
__global__ void k_prep_long(const PrepRange* ranges, int64_t range_cap, int64_t* first_doc, int64_t n_tiles,
                            DevSmall* small) {
  const unsigned long long n_raw = small->n_ranges;
  const unsigned long long n = n_raw < (unsigned long long)range_cap ? n_raw : (unsigned long long)range_cap;
  if (small->status & kStBadInput) return;
  for (unsigned long long r = blockIdx.x; r < n; r += gridDim.x) {
    const PrepRange R = ranges[r];
    const int64_t lo = R.t_lo < 0 ? 0 : R.t_lo, hi = R.t_hi < n_tiles ? R.t_hi : n_tiles - 1;
    for (int64_t t = lo + threadIdx.x; t <= hi; t += blockDim.x) first_doc[t] = R.k;
  }
}

// -------------------------------------------------------- deferred pieces --

// Pre-tokens longer than kShortMax bytes or running past their tile's
// margin, one CTA each (taken from a counter): the end when unknown is the
// first pre-token start of a later tile; the CTA merge (merge_long) leaves
// the ids in the pool at the pre-token's own bytes.
constexpr int kGiantThreads = kThreads;
__global__ void __launch_bounds__(kGiantThreads) k_giants(const uint8_t* bytes, GiantRec* giants, int64_t giant_cap,
                                                          const int64_t* first_start, int64_t n_tiles, TileRec* rec,
                                                          int32_t* pool, Tables T, DevSmall* small) {
  __shared__ int32_t byte_id[256];
  __shared__ uint32_t st_sym[2 * kRound];
  __shared__ uint32_t red[2 * (kThreads / 32)];
  __shared__ uint32_t mred[kThreads / 32];
  __shared__ unsigned long long next;
  __shared__ int64_t end_at;
  const unsigned long long n = small->n_giants < (unsigned long long)giant_cap ? small->n_giants
                                                                               : (unsigned long long)giant_cap;
  if (n == 0) return;
  for (int i = threadIdx.x; i < 256; i += kGiantThreads) byte_id[i] = T.byte_id[i];
  LongScratch L{st_sym, red, mred};
  for (;;) {
    if (threadIdx.x == 0) next = atomicAdd(&small->giant_ctr, 1ull);
    __syncthreads();
    const unsigned long long g = next;
    if (g >= n) break;
    GiantRec R = giants[g];
    if (R.end < 0) {
      // the first tile after R's with a pre-token start holds the end
      if (threadIdx.x == 0) end_at = INT64_MAX;
      __syncthreads();
      for (int64_t t = R.tile + 1; t < n_tiles; t += kGiantThreads) {
        const int64_t tt = t + threadIdx.x;
        const int64_t fs = tt < n_tiles ? first_start[tt] : INT64_MAX;
        if (fs != INT64_MAX) atomicMin(reinterpret_cast<long long*>(&end_at), (long long)fs);
        __syncthreads();
        if (end_at != INT64_MAX) break;
        __syncthreads();
      }
      R.end = end_at;
      if (R.end == INT64_MAX || R.end <= R.start) {
        if (threadIdx.x == 0) atomicOr(&small->status, kStInternal);
        R.end = R.start + 1;
      }
    }
    const uint32_t cnt = merge_long(bytes, R.start, (uint32_t)(R.end - R.start), pool + R.start, T, byte_id, L);
    if (threadIdx.x == 0) {
      giants[g].count = cnt;
      atomicAdd(&rec[R.tile].extra, cnt - 1u);
    }
    __syncthreads();
  }
}

// ----------------------------------------------------------------- output --
// The exclusive offsets of the tiles' final counts (stage entries, less
// holes, plus extra ids) in two levels: k_scan_tiles scans blocks of
// kScanThreads tiles, k_scan_tile_sums (one CTA) the block sums and writes
// the call's token count.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) k_scan_tiles(const TileRec* rec, int64_t n_tiles, uint64_t* tile_base,
                                                             uint64_t* block_sum) {
  __shared__ uint64_t red[kScanThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = blockIdx.x;
  const int64_t t = b * kScanThreads + threadIdx.x;
  uint64_t v = 0;
  if (t < n_tiles) {
    const TileRec R = rec[t];
    v = (uint64_t)R.resv - R.holes + R.extra;
  }
  uint64_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint64_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  uint64_t before = 0, all = 0;
  for (int w = 0; w < kScanThreads / 32; ++w) {
    before += w < warp ? red[w] : 0ull;
    all += red[w];
  }
  if (t < n_tiles) tile_base[t] = before + incl - v;
  if (threadIdx.x == 0) block_sum[b] = all;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_tile_sums(uint64_t* block_sum, int64_t n_blocks,
                                                                 DevSmall* small) {
  __shared__ uint64_t red[kScanThreads / 32];
  __shared__ uint64_t carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int64_t b0 = 0; b0 < n_blocks; b0 += kScanThreads) {
    const int64_t b = b0 + threadIdx.x;
    const uint64_t v = b < n_blocks ? block_sum[b] : 0ull;
    uint64_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint64_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += o;
    }
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    uint64_t before = 0, all = 0;
    for (int w = 0; w < kScanThreads / 32; ++w) {
      before += w < warp ? red[w] : 0ull;
      all += red[w];
    }
    if (b < n_blocks) block_sum[b] = carry + before + incl - v;
    __syncthreads();
    if (threadIdx.x == 0) carry += all;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    small->total = (int64_t)carry;
    small->n_ranges = 0;  // for the next call's k_prep_docs (k_prep_long has read it)
  }
}

constexpr int kCompactWarps = 8;

// What k_compact keeps per tile while it walks the stage.
// A warp per tile: its stage entries to out_ids at the tile's offset without
// the holes, each placeholder given its deferred pre-token's id count (the
// ids are copied from the pool by k_giant_copy). The used part of the tile's
// stage slot is copied to shared memory kCompactPart entries at a time with
// asynchronous 16-byte copies (all loads of a part in flight at once), then
// walked in chunks of 32 entries by one short loop. A chunk of 32 plain ids
// needs no scan; others take positions from a scan of each entry's id count
// (0 for a hole). A document mark (the
// first id of a document) gives document offsets: the r-th mark of the tile
// belongs to the r-th distinct document start in it, which is document k0 + r
// unless the tile has empty documents; then the marks are taken in order and
// each gets the run of documents that start at the same byte as the next
// document not yet placed. The documents at the end of the last one get the
// tile's end.
constexpr int kCompactPart = 512;

__global__ void __launch_bounds__(32 * kCompactWarps, 4) k_compact(const TileRec* rec, const uint32_t* stage,
                                                                const uint64_t* tile_base, const uint64_t* block_sum,
                                                                GiantRec* giants, int64_t giant_cap,
                                                                const int64_t* doc_offsets, int64_t n_tiles,
                                                                int32_t* out_ids, int64_t capacity,
                                                                int64_t* out_offsets, DevSmall* small) {
  __shared__ __align__(16) uint32_t ent_all[kCompactWarps][kCompactPart];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* ent = ent_all[warp];
  const int64_t warps = (int64_t)gridDim.x * kCompactWarps;
  bool over = false;
  int64_t t = (int64_t)blockIdx.x * kCompactWarps + warp;
  // the record and offset of the warp's next tile are loaded a tile ahead
  TileRec Rn{};
  uint64_t base_n = 0;
  if (t < n_tiles) {
    Rn = rec[t];
    base_n = tile_base[t] + block_sum[t / kScanThreads];
  }
  for (; t < n_tiles; t += warps) {
    const TileRec R = Rn;
    const uint32_t* src = stage + t * (int64_t)kTileBits;
    const uint32_t first = min(R.resv, (uint32_t)kCompactPart);
    for (uint32_t c = lane; 4 * c < first; c += 32) cp_async16(ent + 4 * c, src + 4 * c);
    // positions within the tile are 32-bit: at < resv + extra ids of its
    // deferred pre-tokens, ids of the tile's documents k - k0 < 2^31
    const int64_t base = (int64_t)base_n;
    int32_t* out_t = out_ids + base;
    const int64_t room = capacity - base;  // ids of this tile that fit
    const uint32_t cap_t = room <= 0 ? 0u : (room >= (int64_t)UINT32_MAX ? UINT32_MAX : (uint32_t)room);
    int64_t* offs_t = out_offsets + R.k0;
    const uint32_t n_k = (uint32_t)(R.k1 - R.k0);
    if (t + warps < n_tiles) {
      Rn = rec[t + warps];
      base_n = tile_base[t + warps] + block_sum[(t + warps) / kScanThreads];
    }
    uint32_t at0 = 0, nmark = 0;  // the next chunk's first position, document marks so far
    const bool dup = (R.flags & kTileDup) != 0;
    int64_t k_next = R.k0;  // tiles with empty documents: the first document not yet placed
    for (uint32_t p0 = 0; p0 < R.resv; p0 += kCompactPart) {
      const uint32_t n_part = min(R.resv - p0, (uint32_t)kCompactPart);
      if (p0 > 0) {
        __syncwarp();  // the previous part is read
        for (uint32_t c = lane; 4 * c < n_part; c += 32) cp_async16(ent + 4 * c, src + p0 + 4 * c);
      }
      cp_async_wait_all();
      __syncwarp();
      for (uint32_t q0 = 0; q0 < n_part; q0 += 32) {
        const uint32_t e = q0 + lane < n_part ? ent[q0 + lane] : kIdHole;
        const bool plain = (e & kIdSpecial) == 0;  // an id (no hole, no placeholder)
        const uint32_t pb = __ballot_sync(0xFFFFFFFFu, plain);
        uint32_t at = at0 + lane;
        uint32_t n_here = 32;  // ids this chunk places
        bool ph = false;
        if (pb != 0xFFFFFFFFu) {
          const bool valid = (e & (kIdSpecial | kIdLong)) != kIdSpecial;
          const unsigned long long n_giants = small->n_giants;  // records written: min(this, giant_cap)
          ph = valid && !plain && (e & kIdIndex) < n_giants && (e & kIdIndex) < (unsigned long long)giant_cap;
          if (valid && !plain && !ph) atomicOr(&small->status, kStInternal);
          const uint32_t n_ids = (!valid || (!plain && !ph)) ? 0u : (ph ? giants[e & kIdIndex].count : 1u);
          const uint32_t incl = warp_scan_incl(n_ids);
          at = at0 + (incl - n_ids);
          n_here = __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (plain) {
          if (at < cap_t) out_t[at] = (int32_t)(e & ~kIdDoc);
          else over = true;
        }
        const bool mark = (e & kIdDoc) != 0;
        const uint32_t mb = __ballot_sync(0xFFFFFFFFu, mark);
        if (!dup) {
          if (mark) {
            const uint32_t k = nmark + __popc(mb & lanemask_lt());
            if (k < n_k) offs_t[k] = base + at;
            else atomicOr(&small->status, kStInternal);
          }
        } else {
          uint32_t mm = mb;
          while (mm) {  // marks in rank order: each takes the documents at its start
            const int m_lane = __ffs(mm) - 1;
            mm &= mm - 1;
            const int64_t at_m = base + __shfl_sync(0xFFFFFFFFu, at, m_lane);
            const int64_t o0 = k_next < R.k1 ? doc_offsets[k_next] : INT64_MAX;
            int64_t k = k_next;
            while (k < R.k1 && doc_offsets[k] == o0) {
              if (lane == 0) out_offsets[k] = at_m;
              ++k;
            }
            if (k == k_next) atomicOr(&small->status, kStInternal);
            k_next = k;
          }
        }
        uint32_t phm = __ballot_sync(0xFFFFFFFFu, ph);
        while (phm) {
          const int src_lane = __ffs(phm) - 1;
          phm &= phm - 1;
          const uint32_t gv = __shfl_sync(0xFFFFFFFFu, e, src_lane);
          const uint32_t gat = __shfl_sync(0xFFFFFFFFu, at, src_lane);
          if (lane == 0) giants[gv & kIdIndex].at = base + gat;  // k_giant_copy copies its ids
        }
        nmark += __popc(mb);
        at0 += n_here;
      }
    }
    // documents with no mark: at the end of the last document
    const int64_t k_rest = !dup ? R.k0 + nmark : k_next;
    for (int64_t k = k_rest + lane; k < R.k1; k += 32) out_offsets[k] = base + at0;
    __syncwarp();
  }
  if (over) atomicOr(&small->status, kStCapacity);
}

// The ids of the deferred pre-tokens, a CTA each: pool -> out_ids at the
// position k_compact stored, eight loads in flight a thread.
constexpr int kCopyThreads = 256;
__global__ void __launch_bounds__(kCopyThreads) k_giant_copy(const GiantRec* giants, int64_t giant_cap,
                                                               const int32_t* pool, int32_t* out_ids, int64_t capacity,
                                                               DevSmall* small) {
  const unsigned long long n = small->n_giants < (unsigned long long)giant_cap ? small->n_giants
                                                                               : (unsigned long long)giant_cap;
  bool over = false;
  for (unsigned long long g = blockIdx.x; g < n; g += gridDim.x) {
    const int64_t at = giants[g].at;
    const uint32_t count = giants[g].count;
    if (at < 0) continue;
    const int32_t* src = pool + giants[g].start;
    for (uint32_t q0 = 0; q0 < count; q0 += kCopyThreads * 8) {
      int32_t v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t q = q0 + kCopyThreads * u + threadIdx.x;
        v[u] = q < count ? src[q] : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint32_t q = q0 + kCopyThreads * u + threadIdx.x;
        if (q < count) {
          if (at + (int64_t)q < capacity) out_ids[at + q] = v[u];
          else over = true;
        }
      }
    }
  }
  if (over) atomicOr(&small->status, kStCapacity);
}

// ------------------------------------------------------------------ split --
// bpe_pretokenize_batch: the tiles' start bits alone, a warp per tile (no
// workspace: lane 0 finds the tile's first document by binary search).
constexpr int kSplitWarps = 4;
__global__ void __launch_bounds__(32 * kSplitWarps) k_split_tiles(const uint8_t* bytes, int64_t n_bytes,
                                                                  const int64_t* doc_offsets, int64_t n_docs,
                                                                  int64_t n_tiles, uint32_t* out_bits) {
  __shared__ TileWin Wsh[kSplitWarps];
  TileWin& W = Wsh[threadIdx.x >> 5];
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kSplitWarps + (threadIdx.x >> 5);
  if (t >= n_tiles) return;
  const int64_t t0 = t * (int64_t)kTileOwn;
  const bool aligned = (reinterpret_cast<uintptr_t>(bytes) & 15u) == 0;
  tile_load_bytes(W, bytes, n_bytes, t0, aligned);
  int64_t kA = 0;
  if (lane == 0) {
    int64_t lo = 0, hi = n_docs + 1;  // first k with doc_offsets[k] >= t0 - kHalo
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (doc_offsets[mid] < t0 - kHalo) lo = mid + 1;
      else hi = mid;
    }
    kA = lo;
  }
  kA = __shfl_sync(0xFFFFFFFFu, kA, 0);
  int64_t d_first = __ldg(doc_offsets), d_last = __ldg(doc_offsets + n_docs);
  d_first = d_first < 0 ? 0 : (d_first > n_bytes ? n_bytes : d_first);
  d_last = d_last < d_first ? d_first : (d_last > n_bytes ? n_bytes : d_last);
  tile_load_docs(W, doc_offsets, n_docs, t0, kA, d_first, d_last);
  cp_async_wait_all();
  __syncwarp();
  const int64_t n_words = (n_bytes + 31) / 32;
#pragma unroll
  for (int hw = 0; hw < 2; ++hw) {
    const int word = 32 * hw + lane;
    if (word >= kTileWords - 1) continue;  // the margin: the next tile's own bytes
    const int p0 = kHalo + 32 * word;
    uint32_t m;
    if (!ascii_split32(W, p0, &m)) m = start_mask32(W, p0, false);
    const int64_t gw = t0 / 32 + word;
    if (gw < n_words) {
      const int64_t first_bit = gw * 32;
      if (first_bit + 32 > n_bytes) m &= (1u << (n_bytes - first_bit)) - 1u;
      out_bits[gw] = m;
    }
  }
}

}  // namespace
