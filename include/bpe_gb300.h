/*
 * bpe_gb300.h — C ABI of the GB300 batched byte-level BPE encoder.
 *
 * The method (glitch4techs, "Tokenization LLM: building an inference engine
 * in C++", sections "Technical analysis" to "Vocabulary lookup"): split each
 * document into pre-tokens with a GPT-2-style rule, map every UTF-8 byte to
 * its byte-level symbol, repeatedly merge the adjacent pair with the lowest
 * merge rank until no ranked pair remains, and look the resulting symbols up
 * in the vocabulary. A merge step replaces its pair left to right without
 * overlap (tokenwerk, "Tokenisierung", section "Byte Pair Encoding
 * schrittweise") and never crosses a pre-token (dothoosh, "Hugging Face
 * Tokenizers v1 encoding up to 30x", section on how v1 works).
 *
 * Conventions for every call:
 *   - Pointers named d_* are device pointers on the handle's device; h_* are
 *     host pointers. The caller owns every buffer passed in.
 *   - Calls are ordered on the given stream and return once the work is
 *     queued, except where an h_* output is requested: then the call waits
 *     for the stream and also reports errors the kernels detected.
 *   - A handle serves one stream at a time: calls that share a handle must not
 *     overlap on the GPU.
 *   - Return value: BPE_OK, or a BPE_ERR_* code; bpe_last_error() gives a
 *     message (thread-local, valid until the next call on the thread).
 */
#ifndef BPE_GB300_H_
#define BPE_GB300_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BPE_OK 0
#define BPE_ERR_INVALID_ARG 1 /* null pointer, negative size, unknown handle */
#define BPE_ERR_CAPACITY 2    /* an output buffer is too small */
#define BPE_ERR_CUDA 3        /* a CUDA runtime call failed */
#define BPE_ERR_BAD_TABLE 4   /* bpe_build: the merge table or vocabulary is inconsistent */
#define BPE_ERR_TIMEOUT 5     /* a device-side wait gave up (no current kernel waits) */
#define BPE_ERR_INTERNAL 6    /* a device-side consistency check failed */
#define BPE_ERR_BAD_INPUT 7   /* offsets not monotone or outside the buffer, or an id out of range */

typedef struct bpe_handle bpe_handle;
typedef struct CUstream_st* bpe_stream_t; /* a cudaStream_t; NULL = legacy default stream */

/*
 * bpe_build — upload a tokenizer once ("Hugging Face Tokenizers v1", closing
 * section on GPU batch encode: the vocabulary is uploaded once).
 *
 *   merges        host int32[n_merges][3], rows (left_id, right_id, new_id);
 *                 the rank of a row is its index, lower rank merges first
 *                 (glitch4techs, section "Byte Pair Encoding algorithm").
 *   vocab_bytes   host uint8[], the bytes of every token back to back.
 *   vocab_offsets host int64[n_vocab + 1]; token k is
 *                 vocab_bytes[vocab_offsets[k] .. vocab_offsets[k + 1]).
 *                 A token with no bytes is an unused id.
 *   device        CUDA device ordinal that owns the tables.
 *   out           receives the new handle.
 *
 * Checks (BPE_ERR_BAD_TABLE): every one of the 256 single bytes is a token
 * (byte-level base, "Tokenisierung", section "Bytes als robustes Fundament");
 * no two tokens have the same bytes; ids are in [0, n_vocab) and n_vocab <=
 * 2^20; no pair appears twice; bytes(new_id) == bytes(left_id) ||
 * bytes(right_id), so the merged symbol's vocabulary entry is new_id.
 * The handle owns device copies of the tables and a small device workspace.
 */
int bpe_build(const int32_t* merges, int64_t n_merges, const uint8_t* vocab_bytes,
              const int64_t* vocab_offsets, int64_t n_vocab, int device, bpe_handle** out);

/*
 * bpe_encode_batch — encode a batch of documents in one call.
 *
 *   d_bytes        device uint8[n_bytes], the UTF-8 input.
 *   n_bytes        size of d_bytes.
 *   d_doc_offsets  device int64[n_docs + 1]; document k is
 *                  d_bytes[d_doc_offsets[k] .. d_doc_offsets[k + 1]); must be
 *                  non-decreasing within [0, n_bytes]. Empty documents are
 *                  allowed. Bytes outside [d_doc_offsets[0],
 *                  d_doc_offsets[n_docs]) are ignored.
 *   d_out_ids      device int32[out_capacity]; receives the token ids of all
 *                  documents back to back. Tokens never outnumber bytes, so
 *                  out_capacity >= n_bytes always suffices. Ids past
 *                  out_capacity are not written and the call reports
 *                  BPE_ERR_CAPACITY (through h_total_tokens, which then holds
 *                  the count needed, or bpe_sync_status()).
 *   d_out_offsets  device int64[n_docs + 1]; document k's ids are
 *                  d_out_ids[d_out_offsets[k] .. d_out_offsets[k + 1]), with
 *                  d_out_offsets[0] = 0.
 *   h_total_tokens host int64*, may be NULL. When given, the call waits for
 *                  the stream, stores the total token count and returns any
 *                  error found on the device (BPE_ERR_BAD_INPUT, _INTERNAL,
 *                  _CAPACITY). When NULL such errors are kept and returned by
 *                  the next bpe_sync_status() on the handle.
 *   stream         the CUDA stream to run on.
 *
 * Workspace: the handle keeps about 12.7 bytes per input byte:
 *   - a stage of 4.1 bytes per input byte (each 2016-byte tile's ids at their
 *     reserved positions, before the tiles' offsets are known);
 *   - a queue of 4 bytes per input byte for the word-cache misses the tiles
 *     hand to the GPU-wide miss merge (a miss has at least 2 bytes);
 *   - a pool of 4 bytes per input byte (scratch for pre-tokens longer than
 *     64 bytes, each using the range of its own bytes);
 *   - about 56 bytes per tile (first document, record, first pre-token start,
 *     offset) and records of the long pre-tokens (40 bytes each);
 *   - with the per-call memo on (bpe_set_call_memo), 2 bytes per input byte
 *     more and a table of at most 128 MiB.
 * The workspace grows (cudaFree of the old one, then cudaMalloc) the first
 * time a larger batch is seen. No kernel of the call waits on another CTA.
 */
int bpe_encode_batch(bpe_handle* h, const uint8_t* d_bytes, int64_t n_bytes, const int64_t* d_doc_offsets,
                     int64_t n_docs, int32_t* d_out_ids, int64_t out_capacity, int64_t* d_out_offsets,
                     int64_t* h_total_tokens, bpe_stream_t stream);

/*
 * bpe_encode_batch_host — bpe_encode_batch on host buffers. It does the whole
 * round trip and returns when the ids and offsets are in host memory. The
 * pages have no counterpart: the v1 engine of "Hugging Face Tokenizers v1"
 * runs on the CPU.
 *
 * Arguments are those of bpe_encode_batch, but host pointers (h_bytes,
 * h_doc_offsets, h_out_ids, h_out_offsets). Use page-locked memory
 * (cudaMallocHost) for overlap; pageable memory works but copies serialise.
 *
 * Pipeline:
 *   - The batch is cut on document boundaries into slices of about 1/12 of
 *     it (at least 4 MiB); the first and last few are smaller, so encoding
 *     starts and the last copy-out ends soon after the copies start and end.
 *     A document longer than its slice is a slice of its own.
 *   - Slice j's bytes and offsets are copied in on a copy stream of the handle.
 *   - Slice j is encoded on `stream`.
 *   - Slice j-1's ids and offsets are copied out on a second copy stream.
 *   - Four slots of device buffers rotate, so a slice's upload does not wait
 *     on the download of the slice before.
 *
 * Each slice's token count is written by a kernel into page-locked host
 * memory and read on the host before its ids are copied out, so exactly the
 * ids are moved. The offsets are made absolute on the device.
 *
 * Results equal those of bpe_encode_batch on the same batch.
 *
 * Memory: the handle keeps four slots of (slice bytes + 4 B per slice byte +
 * 16 B per slice document) and bpe_encode_batch's workspace for one slice.
 * It grows the first time a larger slice is seen.
 *
 * Errors: BPE_ERR_BAD_INPUT when the first or last offset is outside the
 * buffer or the slice edges are not monotone (checked on the host), and as
 * for bpe_encode_batch otherwise. BPE_ERR_CAPACITY when the ids do not fit
 * (*h_total_tokens then holds the count needed; ids past out_capacity are
 * not written).
 */
int bpe_encode_batch_host(bpe_handle* h, const uint8_t* h_bytes, int64_t n_bytes, const int64_t* h_doc_offsets,
                          int64_t n_docs, int32_t* h_out_ids, int64_t out_capacity, int64_t* h_out_offsets,
                          int64_t* h_total_tokens, bpe_stream_t stream);

/*
 * bpe_encode_batch_noalloc — bpe_encode_batch with fixed scratch: the same
 * arguments, kernels and results, but the call allocates no device memory.
 * The pages have no counterpart; this is a library-level variant for callers
 * that cannot allocate at encode time: a serving loop whose latency cannot
 * absorb the device-wide wait of the cudaFree that bpe_encode_batch issues
 * when its workspace grows, or a process that must fix its device memory
 * footprint before it starts taking requests.
 *
 *   Limit: n_bytes <= 4 MiB (4,194,304). A larger batch is rejected with
 *   BPE_ERR_INVALID_ARG before anything is queued; split it or use
 *   bpe_encode_batch. n_docs is not limited by the scratch.
 *   Scratch: one array of about 53 MB of static device memory per device
 *   (reserved when the library's module is loaded on that device, not by
 *   this call). It holds bpe_encode_batch's workspace for a 4 MiB batch:
 *     - each tile's first document, record, first pre-token start and offset;
 *     - the stage of ids;
 *     - the queue of word-cache misses;
 *     - the records and the pool of long pre-tokens.
 *   The call's first kernel zeroes what must start at zero (the handle's
 *   counters and token count); every other scratch word is written before it
 *   is read.
 *   Set-up: the first call on each device looks up the scratch address
 *   (cudaGetSymbolAddress) and sets the kernels' shared-memory limit, with the
 *   handle's device current; make that first call before any stream capture.
 *   Races: the scratch is shared by every call of this function on a device,
 *   whatever the handle, stream or host thread. Two calls in flight on one
 *   device at the same time overwrite each other's scratch and give wrong ids;
 *   order them on one stream (or wait between them). Calls of bpe_encode_batch
 *   do not touch this scratch.
 * Errors as for bpe_encode_batch. Timing events (bpe_set_timing_events) are
 * not recorded by this call.
 */
int bpe_encode_batch_noalloc(bpe_handle* h, const uint8_t* d_bytes, int64_t n_bytes, const int64_t* d_doc_offsets,
                             int64_t n_docs, int32_t* d_out_ids, int64_t out_capacity, int64_t* d_out_offsets,
                             int64_t* h_total_tokens, bpe_stream_t stream);

/*
 * bpe_pretokenize_batch — the pre-tokenizer alone: marks where pre-tokens
 * start (glitch4techs, section "Technical analysis": the split of "Hello
 * world!" into "Hello", " world", "!").
 *
 *   d_bytes, n_bytes, d_doc_offsets, n_docs   as for bpe_encode_batch.
 *   d_start_bits   device uint32[(n_bytes + 31) / 32]; bit (i % 32) of word
 *                  i / 32 is set iff a pre-token starts at byte i. Every
 *                  non-empty document starts a pre-token; bytes outside the
 *                  documents have no bit set.
 * Needs no handle: the split depends on the text only.
 */
int bpe_pretokenize_batch(const uint8_t* d_bytes, int64_t n_bytes, const int64_t* d_doc_offsets, int64_t n_docs,
                          uint32_t* d_start_bits, bpe_stream_t stream);

/*
 * bpe_decode_batch — token ids back to bytes: the concatenation of every
 * token's bytes ("Tokenisierung", section "Prüfe zuerst den Roundtrip":
 * decode(encode(text)) == text; "Hugging Face Tokenizers v1", section on the
 * road to 1.0: bytes written straight into caller buffers). Byte-exact, no
 * UTF-8 repair.
 *
 *   d_ids             device int32[n_ids].
 *   d_id_offsets      device int64[n_docs + 1], non-decreasing in [0, n_ids].
 *   d_out_bytes       device uint8[out_capacity].
 *   d_out_byte_offsets device int64[n_docs + 1]; document k's bytes are
 *                     d_out_bytes[d_out_byte_offsets[k] .. [k + 1]).
 *   h_total_bytes     host int64*, may be NULL; when given, the call waits and
 *                     stores the byte count; if it exceeds out_capacity the
 *                     call returns BPE_ERR_CAPACITY (nothing past the capacity
 *                     is written).
 * Ids outside [0, n_vocab) decode to nothing and raise BPE_ERR_BAD_INPUT.
 */
int bpe_decode_batch(bpe_handle* h, const int32_t* d_ids, int64_t n_ids, const int64_t* d_id_offsets,
                     int64_t n_docs, uint8_t* d_out_bytes, int64_t out_capacity, int64_t* d_out_byte_offsets,
                     int64_t* h_total_bytes, bpe_stream_t stream);

/*
 * bpe_set_word_cache — turns the handle's word cache on (default) or off.
 * The cache is the memo of "Hugging Face Tokenizers v1" (section on word
 * caching: a given pre-token always yields the same ids, so its ids can be
 * looked up instead of merged). bpe_build fills it once with strings of
 * 2..16 bytes: every vocabulary string, every vocabulary string that starts
 * with a space with the space removed (the word at the start of a line or
 * document), and every prefix of those (a word cut off by the end of a
 * document). Each is run through the device merge loop and its ids (when at
 * most 3) are stored under its bytes. During encoding a pre-token of 2 to 16
 * bytes found there takes the stored ids, a pre-token of one byte is its own
 * token, and every other pre-token runs the merge loop. Either setting gives
 * identical ids.
 */
int bpe_set_word_cache(bpe_handle* h, int enable);

/*
 * bpe_set_call_memo — the per-call memo of the pre-tokens that miss the word
 * cache ("Hugging Face Tokenizers v1", section on word caching: a pre-token
 * always yields the same ids). When it is on, bpe_encode_batch hashes every
 * miss of the call into a table, compares equal hashes byte for byte, merges
 * one pre-token of each distinct string and copies its ids to the others.
 *   BPE_MEMO_AUTO (default): on exactly when the word cache is off (then
 *     every pre-token of two or more bytes is a miss, and they repeat);
 *     with the cache on, the misses are strings the vocabulary does not
 *     hold, nearly all distinct, and the memo would only add work.
 *   BPE_MEMO_ON, BPE_MEMO_OFF: always, never.
 * Either setting gives identical ids. Only bpe_encode_batch uses the memo
 * (bpe_encode_batch_host and bpe_encode_batch_noalloc never do). The memo
 * needs about 2 bytes of workspace per input byte and a table of at most
 * 128 MiB; beyond 2^24 distinct misses the rest are merged one by one.
 * Errors: BPE_ERR_INVALID_ARG for a null handle or another mode.
 */
#define BPE_MEMO_OFF 0
#define BPE_MEMO_ON 1
#define BPE_MEMO_AUTO 2
int bpe_set_call_memo(bpe_handle* h, int mode);

/*
 * bpe_set_timing_events — measurement hook. ev_start and ev_stop are two
 * cudaEvent_t created by the caller on the handle's device. When they are
 * non-NULL, the next bpe_encode_batch calls record them on the call's stream:
 *   - ev_start right before the first kernel;
 *   - ev_stop right after the last kernel.
 * So the caller times all BPE_ENCODE_LAUNCHES kernels of a call together.
 * NULL, NULL switches it off.
 */
int bpe_set_timing_events(bpe_handle* h, void* ev_start, void* ev_stop);

/*
 * bpe_set_phase_events — measurement hook for the time of each kernel.
 * events is an array of BPE_ENCODE_LAUNCHES + 1 cudaEvent_t created by the
 * caller on the handle's device (the handle keeps the pointer, not a copy:
 * the array must outlive its use). While set, bpe_encode_batch records
 * events[0] before its first kernel and events[i] right after its i-th, in
 * this order: k_prep_docs, k_prep_long, k_tiles, k_misses, k_giants,
 * k_scan_tiles, k_scan_tile_sums, k_compact, k_giant_copy (with the per-call
 * memo on, its two kernels run in the k_misses interval). n = 0 (events may
 * be NULL) switches it off; any other n than BPE_ENCODE_LAUNCHES + 1 is
 * BPE_ERR_INVALID_ARG.
 */
#define BPE_ENCODE_LAUNCHES 9
int bpe_set_phase_events(bpe_handle* h, void** events, int n);

/*
 * bpe_train — the merge table of a word list, trained on the GPU
 * ("Tokenisierung", section "Byte Pair Encoding schrittweise": count the
 * adjacent pairs, take the most frequent, ties broken deterministically by
 * the smallest ids, replace it, count again). Byte b is symbol b; merge k
 * makes symbol 256 + k and has rank k. Each step counts every adjacent pair
 * of every word, weighted by the word's count, in a device hash histogram,
 * takes the pair with the largest count (ties: the smallest (left, right)),
 * and replaces it in every word left to right without overlap. Training stops
 * after n_merges merges or when no pair is left.
 *
 *   word_bytes     host uint8, the words back to back (the distinct
 *                  pre-tokens of a corpus).
 *   word_offsets   host int64[n_words + 1], word_offsets[0] = 0,
 *                  non-decreasing.
 *   word_counts    host int64[n_words] >= 0, occurrences of each word.
 *   n_merges       merges wanted (<= 2^20 - 256).
 *   device         CUDA device ordinal; the call allocates, runs on its own
 *                  stream and frees everything before it returns.
 *   merges_out     host int32[n_merges][3]: rows (left, right, new_id).
 *   n_made         host int64*: merges made (<= n_merges).
 * Errors: BPE_ERR_INVALID_ARG for bad arguments, BPE_ERR_CUDA.
 */
int bpe_train(const uint8_t* word_bytes, const int64_t* word_offsets, const int64_t* word_counts, int64_t n_words,
              int64_t n_merges, int device, int32_t* merges_out, int64_t* n_made);

/* Waits for the stream and returns (then clears) errors the kernels of
 * earlier calls on this handle recorded. */
int bpe_sync_status(bpe_handle* h, bpe_stream_t stream);

/* Number of merges and vocabulary size of a handle (host values). */
int bpe_table_info(const bpe_handle* h, int64_t* n_merges, int64_t* n_vocab);

/*
 * bpe_merges_monotone — whether a merge table is monotone: every merge's two
 * operands are single bytes, or ids that a merge of lower rank makes (so a
 * merge can only apply once its operands can exist). A trainer that merges
 * the most frequent pair of the current symbols ("Tokenisierung", section
 * "Byte Pair Encoding schrittweise") always writes monotone tables. On those,
 * replacing every occurrence of the lowest-rank pair per step (this library)
 * and replacing its leftmost occurrence per step give the same ids; on a
 * non-monotone table they can differ (for "abab" with (ab, a) at rank 0 and
 * (a, b) at rank 1 this library gives [ab, ab]).
 *
 *   merges, n_merges, n_vocab   as for bpe_build (host memory).
 *   monotone                    receives 1 or 0.
 * Host-only: needs no GPU and no handle. BPE_ERR_BAD_TABLE for an id outside
 * [0, n_vocab).
 */
int bpe_merges_monotone(const int32_t* merges, int64_t n_merges, int64_t n_vocab, int* monotone);

/* bpe_merges_monotone of the table a handle was built from. */
int bpe_table_monotone(const bpe_handle* h, int* monotone);

/* Bytes of device workspace the handle holds now (0 until a call needs it):
 * bpe_encode_batch, bpe_encode_batch_host and bpe_decode_batch grow it;
 * bpe_encode_batch_noalloc never does. */
int bpe_workspace_bytes(const bpe_handle* h, int64_t* bytes);

/* Frees the handle's device memory. Waits for its device first. */
int bpe_destroy(bpe_handle* h);

/* Message for the last failing call on this thread. */
const char* bpe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* BPE_GB300_H_ */
