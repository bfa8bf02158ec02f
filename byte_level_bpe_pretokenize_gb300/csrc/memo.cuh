// Per-call memo of the word-cache misses ("Hugging Face Tokenizers v1",
// section "word caching mechanism": a pre-token always gives the same ids,
// so a repeated one need not be merged again), for calls where the misses
// repeat (the word cache off: every pre-token of two or more bytes is a miss).
//
// Included once by bpe_kernels.cu after tiles.cuh; not a standalone header.
//
//   * k_memo_claim (after k_tiles): a thread per queued miss hashes its bytes
//     and claims a slot of an open-addressed table (tag << 32 | queue index,
//     atomicCAS). A slot already holding the same tag is compared byte for
//     byte with that owner's pre-token; an equal one makes this miss its
//     follower. A miss that finds no slot within kMemoProbes merges itself.
//   * k_misses merges the owners only (followers read as empty entries).
//   * k_memo_copy (after k_misses): a thread per follower copies its owner's
//     reserved stage entries (ids, then holes) to its own reservation, with
//     its own document mark, and adds its holes to its tile's record.
// The host empties the table (a memset) before k_memo_claim in every call.

namespace {

constexpr uint64_t kMemoEmpty = ~0ull;
constexpr int kMemoProbes = 64;
constexpr int kMemoThreads = 256;

__device__ __forceinline__ const uint8_t* miss_src(const uint8_t* bytes, uint64_t e) {
  return bytes + (int64_t)(e >> 30) * kTileOwn + (int64_t)(e & 0x7FFu);
}
__device__ __forceinline__ uint32_t miss_len(uint64_t e) { return (uint32_t)(e >> kMissLenShift) & 0x7Fu; }

__global__ void __launch_bounds__(kMemoThreads) k_memo_claim(const uint8_t* bytes, const uint64_t* queue,
                                                             int64_t queue_cap, uint64_t* table, uint64_t mask,
                                                             uint32_t* follow, DevSmall* small) {
  const unsigned long long n_raw = small->n_misses;
  const uint64_t n_q = n_raw < (unsigned long long)queue_cap ? n_raw : (unsigned long long)queue_cap;
  for (uint64_t q = (uint64_t)blockIdx.x * kMemoThreads + threadIdx.x; q < n_q;
       q += (uint64_t)gridDim.x * kMemoThreads) {
    const uint64_t e = queue[q];
    const uint32_t n = miss_len(e);
    const uint8_t* src = miss_src(bytes, e);
    uint32_t h = 0x811C9DC5u ^ n;
    for (uint32_t i = 0; i < n; ++i) h = (h ^ src[i]) * 0x01000193u;  // FNV-1a 32 over the bytes
    const uint32_t tag = mix32(h) | 1u;
    uint64_t slot = (uint64_t)h & mask;
    uint32_t owner = (uint32_t)q;
    for (int probe = 0; probe < kMemoProbes; ++probe, slot = (slot + 1) & mask) {
      uint64_t cur = table[slot];
      if (cur == kMemoEmpty) {
        cur = atomicCAS(reinterpret_cast<unsigned long long*>(table + slot), (unsigned long long)kMemoEmpty,
                        (unsigned long long)tag << 32 | (unsigned long long)q);
        if (cur == kMemoEmpty) break;  // claimed: this miss is the owner
      }
      if ((uint32_t)(cur >> 32) != tag) continue;
      const uint32_t o = (uint32_t)cur;
      const uint64_t eo = queue[o];
      if (miss_len(eo) != n) continue;
      const uint8_t* so = miss_src(bytes, eo);
      bool same = true;
      for (uint32_t i = 0; i < n && same; ++i) same = so[i] == src[i];
      if (same) {
        owner = o;
        break;
      }
    }
    follow[q] = owner;
  }
}

__global__ void __launch_bounds__(kMemoThreads) k_memo_copy(const uint64_t* queue, int64_t queue_cap,
                                                            const uint32_t* follow, uint32_t* stage, TileRec* rec,
                                                            DevSmall* small) {
  const unsigned long long n_raw = small->n_misses;
  const uint64_t n_q = n_raw < (unsigned long long)queue_cap ? n_raw : (unsigned long long)queue_cap;
  for (uint64_t q = (uint64_t)blockIdx.x * kMemoThreads + threadIdx.x; q < n_q;
       q += (uint64_t)gridDim.x * kMemoThreads) {
    const uint32_t o = follow[q];
    if (o == (uint32_t)q || o >= n_q) continue;
    const uint64_t e = queue[q], eo = queue[o];
    const uint32_t n = miss_len(e);
    const uint32_t* src = stage + (int64_t)(eo >> 30) * kTileBits + ((eo >> kMissAtShift) & 0x7FFu);
    uint32_t* dst = stage + (int64_t)(e >> 30) * kTileBits + ((e >> kMissAtShift) & 0x7FFu);
    const uint32_t doc = ((e >> kMissDocShift) & 1u) ? kIdDoc : 0u;
    uint32_t holes = 0;
    for (uint32_t i = 0; i < n; ++i) {
      uint32_t v = src[i];
      if (i == 0) v = (v & ~kIdDoc) | doc;
      holes += (v & kIdSpecial) ? 1u : 0u;
      dst[i] = v;
    }
    if (holes) atomicAdd(&rec[(int64_t)(e >> 30)].holes, holes);
  }
}

}  // namespace
