// Training: the merge table from a word list ("Tokenisierung", section "Byte
// Pair Encoding schrittweise": count the adjacent pairs, take the most
// frequent, ties to the smallest ids, replace it everywhere, count again).
//
// Included once by bpe_kernels.cu; not a standalone header.
//
// The words are the distinct pre-tokens of a corpus with their counts. Byte b
// starts as symbol b; merge k makes symbol 256 + k and has rank k. One step,
// all on the device and without a host round trip:
//   * k_train_count: a thread per word adds the word's count to every
//     adjacent pair of its symbols in an open-addressed pair histogram
//     (64-bit key left << 32 | right, 64-bit count; atomicCAS claims a slot,
//     and a claimed slot is listed, so the other two kernels touch only the
//     pairs that occur).
//   * k_train_best: the most frequent listed pair, ties to the smallest
//     (left, right): block reductions, then the last CTA to finish reduces
//     the block results and appends the merge row. With no pair left it sets
//     the done flag and later steps return at once.
//   * k_train_replace: a thread per word replaces the pair left to right
//     without overlap and compacts the word in place; it also empties the
//     listed slots for the next step.
// Every step is the same three launches with the same arguments, so the host
// captures a run of steps in a CUDA graph once and replays it.

namespace {

constexpr uint64_t kTrainEmpty = ~0ull;
constexpr int kTrainThreads = 256;
constexpr int kTrainLocal = 2048;  // claimed slots a CTA lists in shared memory

struct TrainState {
  unsigned long long best_count;
  unsigned long long best_key;
  unsigned int blocks_done;
  int done;        // no pair left, or n_merges made: later steps return at once
  int merged_now;  // this step made a merge (k_train_replace applies it)
  long long made;
  unsigned long long n_occ;    // histogram slots claimed in this step (listed in occ)
  unsigned long long n_clear;  // slots k_train_replace empties (this step's n_occ)
};

__device__ __forceinline__ uint32_t train_hash(uint64_t k) {
  return mix32((uint32_t)k * 0x9E3779B1u ^ mix32((uint32_t)(k >> 32)));
}

// (count, key) order: larger count first, then smaller key.
__device__ __forceinline__ bool train_better(uint64_t c1, uint64_t k1, uint64_t c2, uint64_t k2) {
  return c1 > c2 || (c1 == c2 && k1 < k2);
}

__global__ void __launch_bounds__(kTrainThreads) k_train_count(const int32_t* sym, const int64_t* off,
                                                               const int32_t* len, const int64_t* freq,
                                                               int64_t n_words, uint64_t* keys,
                                                               unsigned long long* counts, uint64_t mask,
                                                               uint32_t* occ, TrainState* st) {
  // slots this CTA claims, listed in shared memory and appended to occ with
  // one global atomic at the end (past kTrainLocal, one atomic each)
  __shared__ uint32_t loc[kTrainLocal];
  __shared__ unsigned int n_loc;
  __shared__ unsigned long long base;
  if (st->done) return;
  if (threadIdx.x == 0) n_loc = 0;
  __syncthreads();
  for (int64_t w = (int64_t)blockIdx.x * kTrainThreads + threadIdx.x; w < n_words;
       w += (int64_t)gridDim.x * kTrainThreads) {
    const int32_t* s = sym + off[w];
    const int32_t n = len[w];
    const unsigned long long f = (unsigned long long)freq[w];
    for (int32_t i = 0; i + 1 < n; ++i) {
      const uint64_t key = (uint64_t)(uint32_t)s[i] << 32 | (uint32_t)s[i + 1];
      uint64_t h = train_hash(key) & mask;
      for (uint64_t probe = 0; probe <= mask; ++probe) {
        const unsigned long long prev =
            atomicCAS(reinterpret_cast<unsigned long long*>(keys + h), (unsigned long long)kTrainEmpty,
                      (unsigned long long)key);
        if (prev == kTrainEmpty || prev == key) {
          if (prev == kTrainEmpty) {
            const unsigned int j = atomicAdd(&n_loc, 1u);
            if (j < (unsigned)kTrainLocal) loc[j] = (uint32_t)h;
            else occ[atomicAdd(&st->n_occ, 1ull)] = (uint32_t)h;
          }
          atomicAdd(counts + h, f);
          break;
        }
        h = (h + 1) & mask;
      }
    }
  }
  __syncthreads();
  const unsigned int n = n_loc < (unsigned)kTrainLocal ? n_loc : (unsigned)kTrainLocal;
  if (threadIdx.x == 0) base = n ? atomicAdd(&st->n_occ, (unsigned long long)n) : 0ull;
  __syncthreads();
  for (unsigned int j = threadIdx.x; j < n; j += kTrainThreads) occ[base + j] = loc[j];
}

__global__ void __launch_bounds__(kTrainThreads) k_train_best(const uint64_t* keys, const unsigned long long* counts,
                                                              const uint32_t* occ, unsigned long long* block_count,
                                                              unsigned long long* block_key, TrainState* st,
                                                              int32_t* merges, int64_t n_merges) {
  __shared__ unsigned long long sc[kTrainThreads / 32], sk[kTrainThreads / 32];
  __shared__ bool last;
  if (st->done) return;
  const uint64_t n_occ = st->n_occ;
  uint64_t bc = 0, bk = kTrainEmpty;
  for (uint64_t j = (uint64_t)blockIdx.x * kTrainThreads + threadIdx.x; j < n_occ;
       j += (uint64_t)gridDim.x * kTrainThreads) {
    const uint32_t i = occ[j];
    const uint64_t k = keys[i];
    const uint64_t c = counts[i];
    if (train_better(c, k, bc, bk)) {
      bc = c;
      bk = k;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const uint64_t oc = __shfl_xor_sync(0xFFFFFFFFu, bc, d), ok = __shfl_xor_sync(0xFFFFFFFFu, bk, d);
    if (train_better(oc, ok, bc, bk)) {
      bc = oc;
      bk = ok;
    }
  }
  if (lane == 0) {
    sc[warp] = bc;
    sk[warp] = bk;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kTrainThreads / 32; ++w)
      if (train_better(sc[w], sk[w], bc, bk)) {
        bc = sc[w];
        bk = sk[w];
      }
    block_count[blockIdx.x] = bc;
    block_key[blockIdx.x] = bk;
    __threadfence();
    last = atomicAdd(&st->blocks_done, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last || warp != 0) return;
  // the last CTA's first warp: every block result is visible (each was
  // fenced before its counter increment)
  __threadfence();
  bc = 0;
  bk = kTrainEmpty;
  for (unsigned b = lane; b < gridDim.x; b += 32) {
    const uint64_t c = *reinterpret_cast<volatile unsigned long long*>(block_count + b);
    const uint64_t k = *reinterpret_cast<volatile unsigned long long*>(block_key + b);
    if (train_better(c, k, bc, bk)) {
      bc = c;
      bk = k;
    }
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const uint64_t oc = __shfl_xor_sync(0xFFFFFFFFu, bc, d), ok = __shfl_xor_sync(0xFFFFFFFFu, bk, d);
    if (train_better(oc, ok, bc, bk)) {
      bc = oc;
      bk = ok;
    }
  }
  if (lane != 0) return;
  st->blocks_done = 0;
  st->merged_now = 0;
  st->n_clear = st->n_occ;  // every CTA has read n_occ
  st->n_occ = 0;
  if (bc == 0 || st->made >= n_merges) {
    st->done = 1;
    return;
  }
  const long long m = st->made;
  merges[3 * m] = (int32_t)(bk >> 32);
  merges[3 * m + 1] = (int32_t)(uint32_t)bk;
  merges[3 * m + 2] = 256 + (int32_t)m;
  st->best_count = bc;
  st->best_key = bk;
  st->made = m + 1;
  st->merged_now = 1;
}

__global__ void __launch_bounds__(kTrainThreads) k_train_replace(int32_t* sym, const int64_t* off, int32_t* len,
                                                                 int64_t n_words, uint64_t* keys,
                                                                 unsigned long long* counts, const uint32_t* occ,
                                                                 const TrainState* st) {
  // the slots this step claimed are emptied for the next step
  const uint64_t n_clear = st->n_clear;
  for (uint64_t j = (uint64_t)blockIdx.x * kTrainThreads + threadIdx.x; j < n_clear;
       j += (uint64_t)gridDim.x * kTrainThreads) {
    const uint32_t i = occ[j];
    keys[i] = kTrainEmpty;
    counts[i] = 0;
  }
  if (!st->merged_now) return;  // no merge was made by this step
  const int32_t a = (int32_t)(st->best_key >> 32), b = (int32_t)(uint32_t)st->best_key;
  const int32_t nw = 256 + (int32_t)(st->made - 1);
  for (int64_t w = (int64_t)blockIdx.x * kTrainThreads + threadIdx.x; w < n_words;
       w += (int64_t)gridDim.x * kTrainThreads) {
    int32_t* s = sym + off[w];
    const int32_t n = len[w];
    int32_t m = 0;
    for (int32_t i = 0; i < n;) {
      if (i + 1 < n && s[i] == a && s[i + 1] == b) {
        s[m++] = nw;
        i += 2;
      } else {
        s[m++] = s[i++];
      }
    }
    len[w] = m;
  }
}

}  // namespace
