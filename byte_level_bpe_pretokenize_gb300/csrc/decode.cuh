// Decoding: token ids back to bytes ("Tokenisierung", section "Prüfe zuerst
// den Roundtrip": decode(encode(text)) == text; the bytes of a token are its
// vocabulary string, section "Bytes als robustes Fundament").
//
// Included once by bpe_kernels.cu; not a standalone header.
//
// The ids are cut into tiles of kDecIds. Per call:
//   * k_dec_count: a warp per tile sums its tokens' byte lengths.
//   * k_dec_scan_tiles, then k_scan_tile_sums: exclusive byte offsets of the
//     tiles and the call's total.
//   * k_dec_first_doc: a thread per tile finds the first document whose id
//     offset is at or past the tile's first id (a binary search), and the
//     document offsets are validated.
//   * k_dec_write: a warp per tile places its tokens' bytes in shared memory
//     at the tile's output alignment (buffer index = output address mod 16)
//     and stores them with 16-byte stores; the documents that start in the
//     tile get their byte offsets from the same warp scan.
// Token entries (bpe_build): the first 12 bytes of the token and its length,
// one 16-byte load; longer tokens read the rest from the vocabulary bytes.

namespace {

constexpr int kDecIds = 1024;          // ids per tile
constexpr int kDecWarps = 8;           // tiles in flight per CTA
constexpr int kDecBuf = 8192;          // bytes a warp buffers before it stores them
constexpr int kDecScanThreads = 1024;  // tiles per block of the tile scan
constexpr uint32_t kDecInline = 12;    // token bytes held in its entry
constexpr int kDecAhead = 4;           // rounds of 32 ids whose loads are issued together

__device__ __forceinline__ uint4 dec_entry(const uint4* vent, int64_t n_vocab, int32_t id, bool* bad) {
  if (id < 0 || (int64_t)id >= n_vocab) {
    *bad = true;
    return make_uint4(0, 0, 0, 0);
  }
  return __ldg(vent + id);
}

__global__ void __launch_bounds__(32 * kDecWarps) k_dec_count(const int32_t* ids, int64_t n_ids, const uint4* vent,
                                                              int64_t n_vocab, int64_t n_tiles, uint64_t* tile_bytes,
                                                              DevSmall* small) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
  for (int64_t t = (int64_t)blockIdx.x * kDecWarps + (threadIdx.x >> 5); t < n_tiles;
       t += (int64_t)gridDim.x * kDecWarps) {
    const int64_t i0 = t * kDecIds;
    const int64_t n = n_ids - i0 < kDecIds ? n_ids - i0 : kDecIds;
    uint32_t sum = 0;
    for (int j0 = 0; j0 < kDecIds / 32; j0 += 8) {  // eight ids, then their eight entries, in flight
      int32_t id[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t i = (int64_t)(j0 + u) * 32 + lane;
        id[u] = i < n ? __ldcs(ids + i0 + i) : -1;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if ((int64_t)(j0 + u) * 32 + lane < n) sum += dec_entry(vent, n_vocab, id[u], &bad).w;
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, d);
    if (lane == 0) tile_bytes[t] = sum;
  }
  if (bad) atomicOr(&small->status, kStBadInput);
}

// Exclusive scan of tile_bytes in place over blocks of kDecScanThreads tiles;
// block sums to block_sum (scanned by k_scan_tile_sums).
__global__ void __launch_bounds__(kDecScanThreads) k_dec_scan_tiles(uint64_t* tile_bytes, int64_t n_tiles,
                                                                    uint64_t* block_sum) {
  __shared__ uint64_t red[kDecScanThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t t = (int64_t)blockIdx.x * kDecScanThreads + threadIdx.x;
  const uint64_t v = t < n_tiles ? tile_bytes[t] : 0ull;
  uint64_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint64_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += o;
  }
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  uint64_t before = 0, all = 0;
  for (int w = 0; w < kDecScanThreads / 32; ++w) {
    before += w < warp ? red[w] : 0ull;
    all += red[w];
  }
  if (t < n_tiles) tile_bytes[t] = before + incl - v;
  if (threadIdx.x == 0) block_sum[blockIdx.x] = all;
}

// first_doc[t] = the first k with id_offsets[k] >= t * kDecIds (n_docs + 1 if
// none); thread k <= n_docs also checks document k's offset.
__global__ void k_dec_first_doc(const int64_t* id_offsets, int64_t n_docs, int64_t n_ids, int64_t n_tiles,
                                int64_t* first_doc, DevSmall* small) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  bool bad = false;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n_tiles || x <= n_docs; x += stride) {
    if (x <= n_docs) {
      const int64_t o = __ldg(id_offsets + x);
      if (o < 0 || o > n_ids || (x > 0 && o < __ldg(id_offsets + x - 1))) bad = true;
    }
    if (x < n_tiles) {
      const int64_t want = x * kDecIds;
      int64_t lo = 0, hi = n_docs + 1;
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (__ldg(id_offsets + mid) < want) lo = mid + 1;
        else hi = mid;
      }
      first_doc[x] = lo;
    }
  }
  if (bad) atomicOr(&small->status, kStBadInput);
}

// The warp's buffer bytes [lo, hi) go to out + g0 + (b - lo) for buffer index
// b, where (out + g0) mod 16 == lo mod 16: whole 16-byte chunks with one
// store, the two edge chunks byte by byte; nothing at or past cap.
__device__ __forceinline__ bool dec_flush(const uint8_t* buf, uint32_t lo, uint32_t hi, uint8_t* out, int64_t g0,
                                          int64_t cap) {
  const uint32_t lane = threadIdx.x & 31u;
  bool over = false;
  if (hi <= lo) return false;
  const bool room = g0 + (int64_t)(hi - lo) <= cap;
  uint8_t* dst = out + g0;  // buffer index b -> dst[b - lo]; whole chunks are 16-byte aligned there
  for (uint32_t c = (lo >> 4) + lane; c <= ((hi - 1) >> 4); c += 32) {
    const uint32_t b0 = c << 4;
    if (room && b0 >= lo && b0 + 16 <= hi) {
      *reinterpret_cast<uint4*>(dst + (b0 - lo)) = *reinterpret_cast<const uint4*>(buf + b0);
    } else {
      for (uint32_t b = b0 < lo ? lo : b0; b < b0 + 16 && b < hi; ++b) {
        if (g0 + (int64_t)(b - lo) < cap) dst[b - lo] = buf[b];
        else over = true;
      }
    }
  }
  return over;
}

__global__ void __launch_bounds__(32 * kDecWarps) k_dec_write(const int32_t* ids, int64_t n_ids, const uint4* vent,
                                                              const uint8_t* vbytes, const int64_t* voffs,
                                                              int64_t n_vocab, const uint64_t* tile_base,
                                                              const uint64_t* block_sum, const int64_t* first_doc,
                                                              const int64_t* id_offsets, int64_t n_docs,
                                                              int64_t n_tiles, uint8_t* out, int64_t cap,
                                                              int64_t* out_offsets, DevSmall* small) {
  __shared__ __align__(16) uint8_t buf_all[kDecWarps][kDecBuf + 32];
  uint8_t* buf = buf_all[threadIdx.x >> 5];
  const uint32_t lane = threadIdx.x & 31u;
  bool over = false, bad = false;
  for (int64_t t = (int64_t)blockIdx.x * kDecWarps + (threadIdx.x >> 5); t < n_tiles;
       t += (int64_t)gridDim.x * kDecWarps) {
    const int64_t i0 = t * kDecIds;
    const int64_t n = n_ids - i0 < kDecIds ? n_ids - i0 : kDecIds;
    const int64_t base = (int64_t)(tile_base[t] + block_sum[t / kDecScanThreads]);
    const bool last = t == n_tiles - 1;
    // the documents of the tile, 32 at a time: lane l holds document kb + l
    int64_t kb = first_doc[t];
    int64_t doff = kb + lane <= n_docs ? __ldg(id_offsets + kb + lane) : INT64_MAX;
    // buffer: index b holds output byte g_lo + (b - lo); (out + g_lo) mod 16 == lo mod 16
    int64_t g_lo = base;
    uint32_t lo = (uint32_t)(reinterpret_cast<uintptr_t>(out + base) & 15u), hi = lo;
    int64_t at = base;  // output position of the next token
    for (int64_t g0 = 0; g0 < n; g0 += 32 * kDecAhead) {
     // the ids and token entries of kDecAhead rounds are loaded together
     int32_t idg[kDecAhead];
     uint4 eg[kDecAhead];
#pragma unroll
     for (int u = 0; u < kDecAhead; ++u) {
       const int64_t i = g0 + 32 * u + lane;
       idg[u] = i < n ? __ldcs(ids + i0 + i) : -1;
     }
#pragma unroll
     for (int u = 0; u < kDecAhead; ++u)
       eg[u] = g0 + 32 * u + lane < n ? dec_entry(vent, n_vocab, idg[u], &bad) : make_uint4(0, 0, 0, 0);
     // the group's kDecAhead scans together (independent chains)
     uint32_t len[kDecAhead], incl[kDecAhead];
#pragma unroll
     for (int u = 0; u < kDecAhead; ++u) incl[u] = len[u] = eg[u].w;
#pragma unroll
     for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
       for (int u = 0; u < kDecAhead; ++u) {
         const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, incl[u], d);
         if (lane >= (uint32_t)d) incl[u] += o;
       }
     }
     uint32_t gb[kDecAhead];  // bytes of the group's rounds before round u
     uint32_t gtot = 0;
#pragma unroll
     for (int u = 0; u < kDecAhead; ++u) {
       gb[u] = gtot;
       gtot += __shfl_sync(0xFFFFFFFFu, incl[u], 31);
     }
     // documents whose first id is in the group: the byte offset of that id
     const int64_t gn = n - g0 < 32 * kDecAhead ? n - g0 : 32 * kDecAhead;  // ids of the group
     for (;;) {
       const int64_t rel = doff - (i0 + g0);
       const bool here = rel >= 0 && rel < gn;
       const uint32_t src = here ? (uint32_t)(rel & 31) : lane;
       uint32_t pre = 0;
#pragma unroll
       for (int u = 0; u < kDecAhead; ++u) {
         const uint32_t x = __shfl_sync(0xFFFFFFFFu, incl[u] - len[u], src);
         if (here && (rel >> 5) == u) pre = gb[u] + x;
       }
       if (here) out_offsets[kb + lane] = at + pre;
       const bool done = doff == INT64_MAX || rel < gn;
       if (!__all_sync(0xFFFFFFFFu, done) || kb + 32 > n_docs) break;
       kb += 32;
       doff = kb + lane <= n_docs ? __ldg(id_offsets + kb + lane) : INT64_MAX;
     }
     // bytes: flush first when the group does not fit; a group larger than
     // the buffer goes straight to the output
     if (hi + gtot > (uint32_t)kDecBuf) {
       __syncwarp();
       over |= dec_flush(buf, lo, hi, out, g_lo, cap);
       __syncwarp();
       g_lo = at;
       lo = hi = (uint32_t)(reinterpret_cast<uintptr_t>(out + at) & 15u);
     }
     const bool direct = hi + gtot > (uint32_t)kDecBuf;
#pragma unroll
     for (int u = 0; u < kDecAhead; ++u) {
       const uint4 e = eg[u];
       const uint32_t L = len[u], off = gb[u] + incl[u] - L;
       if (direct) {
         const int64_t b0 = L > kDecInline ? voffs[idg[u]] : 0;
         for (uint32_t q = 0; q < L; ++q) {
           const int64_t g = at + off + q;
           const uint8_t v = q < kDecInline ? (uint8_t)((q < 4 ? e.x : q < 8 ? e.y : e.z) >> (8 * (q & 3))) : vbytes[b0 + q];
           if (g < cap) out[g] = v;
           else over = true;
         }
       } else {
         uint8_t* d = buf + hi + off;
#pragma unroll
         for (uint32_t q = 0; q < kDecInline; ++q)
           if (q < L) d[q] = (uint8_t)((q < 4 ? e.x : q < 8 ? e.y : e.z) >> (8 * (q & 3)));
         if (L > kDecInline) {
           const uint8_t* src = vbytes + voffs[idg[u]];
           for (uint32_t q = kDecInline; q < L; ++q) d[q] = src[q];
         }
       }
     }
     if (direct) {
       g_lo = at + gtot;
       lo = hi = (uint32_t)(reinterpret_cast<uintptr_t>(out + g_lo) & 15u);
     } else {
       hi += gtot;
     }
     at += gtot;
    }
    __syncwarp();
    over |= dec_flush(buf, lo, hi, out, g_lo, cap);
    __syncwarp();
    if (last) {  // documents that start at the end of the ids
      for (;;) {
        if (doff == n_ids) out_offsets[kb + lane] = at;
        if (!__all_sync(0xFFFFFFFFu, doff <= n_ids || doff == INT64_MAX) || kb + 32 > n_docs) break;
        kb += 32;
        doff = kb + lane <= n_docs ? __ldg(id_offsets + kb + lane) : INT64_MAX;
      }
    }
  }
  if (over) atomicOr(&small->status, kStCapacity);
  if (bad) atomicOr(&small->status, kStBadInput);
}

}  // namespace
