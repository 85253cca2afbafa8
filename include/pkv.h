/*
 * pkv.h -- C ABI of the paged KV-cache decode library (GB300, sm_103a).
 *
 * Two operations make up one decode step of one attention layer over a block-paged
 * KV cache:
 *
 *   pkv_paged_kv_append         scatter the step's new K/V rows into the pool
 *   pkv_paged_decode_attention  one query vector per sequence attends over that
 *                               sequence's cached K/V, gathered through its block table
 *
 * Sources (page title, section):
 *   habr.com/ru/articles/1021832 ("KV-Cache ... в рамках одного GPU"):
 *     section 1 "Prefill и Decode"  -- decode appends one new K,V per step ("append");
 *     section 2 "KV-Cache: цена памяти" -- bytes/token formula, GQA (query heads
 *        sharing a KV head), FP8 KV cache (--kv-cache-dtype fp8);
 *     section 3 "Вспомним FlashAttention" -- Attention(Q,K,V) = softmax(QK^T/sqrt(d_k))V,
 *        computed tile by tile with a running max and running sum, exactly;
 *     section 4 "Вспомним PagedAttention" -- 16-token blocks, block table as a page
 *        table, blocks scattered in GPU memory, worked example of slot assignment;
 *     section 5 "Как vLLM объединяет FlashAttention и PagedAttention" -- the decode call
 *        flash_attn_with_kvcache(q [batch,1,num_heads,d_head],
 *        k_cache/v_cache [num_physical_blocks, block_size, num_kv_heads, d_head],
 *        block_table [batch, max_num_blocks] int32, cache_seqlens [batch]).
 *   actionbridge.io ... chapter 8 "KV cache management" -- flat physical pool, the
 *     attention kernel gathers keys and values through the block table.
 *
 * Conventions shared by every call
 *   - All data pointers are DEVICE pointers on the current CUDA device, owned by the
 *     caller.  The library allocates no device or pinned memory and keeps no state
 *     except cached device properties, a cached driver entry point, a device status
 *     word (see pkv_check_device_status) and a thread-local error string.
 *   - Calls enqueue work on `stream` and return without synchronising.  A NULL stream
 *     is the legacy default stream.
 *   - Host-side validation runs before anything is enqueued; on failure nothing is
 *     enqueued and the call returns PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED /
 *     PKV_ERR_WORKSPACE with a message in pkv_last_error().  A failed launch returns
 *     PKV_ERR_CUDA.  No C++ exception crosses this interface.
 *   - Data-dependent checks run on the device without faulting: a slot outside the
 *     pool, a block id outside the pool, a context length outside
 *     [0, min(max_context_len, max_blocks_per_seq*16)] are skipped or clamped, and a
 *     bit is set in the device status word, which pkv_check_device_status reports.
 *     Reads through an out-of-range block id return zeros (the tensor-map bounds of the
 *     pool), never memory outside it.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, declared here so C callers need no CUDA header. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,  /* bad pointer, shape, alignment or size */
  PKV_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head_dim, group size, device) */
  PKV_ERR_WORKSPACE = 3,    /* workspace missing or smaller than pkv_decode_workspace_size() */
  PKV_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  PKV_ERR_DEVICE_CHECK = 5  /* pkv_check_device_status found a device-side check failure */
} pkv_status;

typedef enum {
  PKV_KV_BF16 = 0,     /* pool elements are bf16 */
  PKV_KV_FP8_E4M3 = 1  /* pool elements are OCP E4M3 bytes with per-(K|V, kv head) fp32 scales */
} pkv_kv_dtype;

typedef enum { PKV_OUT_BF16 = 0, PKV_OUT_FP32 = 1 } pkv_out_dtype;

/* Device status word bits (pkv_check_device_status). */
#define PKV_DEVFLAG_BAD_SLOT 0x1u        /* append: slot >= num_blocks * block_size (skipped) */
#define PKV_DEVFLAG_BAD_CONTEXT_LEN 0x2u /* decode: context length out of range (clamped) */
#define PKV_DEVFLAG_BAD_BLOCK_ID 0x4u    /* decode: block id outside the pool (read as zeros);
                                            copy: pair skipped */
#define PKV_DEVFLAG_WAIT_TIMEOUT 0x8u    /* decode: a pipeline wait hit its iteration limit */

/*
 * The caller-owned paged pool.  Nothing is copied; the struct is read during the call.
 *   k_cache, v_cache: [num_blocks][block_size][num_kv_heads][head_dim], row-major,
 *     elements bf16 (2 bytes) or E4M3 (1 byte) -- the layout of section 5 above.
 *     Both must be 16-byte aligned.  num_blocks * block_size must fit in int32.
 *   block_size: must be 16 (section 4: "по умолчанию — 16").
 *   head_dim: 64 or 128.
 *   scales: for PKV_KV_FP8_E4M3, device fp32 [2][num_kv_heads] -- row 0 scales K, row 1
 *     scales V; a stored code c means the value decode(c) * scale.  NULL for bf16.
 */
typedef struct {
  void* k_cache;
  void* v_cache;
  int64_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  pkv_kv_dtype kv_dtype;
  const float* scales;
} pkv_cache_desc;

/*
 * Append one step's new K/V rows (section 1 "append", section 4 worked example: token
 * 1025 goes to the next free slot of the sequence's current block).
 *   k, v: [num_tokens][num_kv_heads][head_dim] bf16, 16-byte aligned.
 *   slot_mapping: [num_tokens] int64; slot = physical_block * block_size + offset.
 *     slot < 0 skips the token (padding).  slot >= num_blocks*block_size is skipped and
 *     sets PKV_DEVFLAG_BAD_SLOT.
 *   For every kept token t, head h, element i:
 *     cache[slot / block_size][slot % block_size][h][i] = enc(x[t][h][i])
 *   where enc is a bit copy for bf16, and for E4M3 the binary32 division x / scale
 *   (scale = scales[0][h] for K, scales[1][h] for V) rounded to nearest-even E4M3 and
 *   saturated to +-448.
 *   Two tokens with the same slot: which one lands is unspecified.
 *   num_tokens == 0 is a no-op returning PKV_OK.
 */
pkv_status pkv_paged_kv_append(const pkv_cache_desc* cache, const void* k, const void* v,
                               const int64_t* slot_mapping, int64_t num_tokens,
                               pkv_stream_t stream);

/*
 * Copy whole blocks of the pool (copy-on-write; section 4, "Copy-on-Write": sequences that
 * share a block through reference counts get their own copy before one of them writes into
 * it, the original staying untouched).
 *   block_pairs: [num_pairs][2] int64 device array of (src, dst) physical block ids.  For
 *   each pair, block dst of k_cache and of v_cache becomes a bit copy of block src (all
 *   block_size slots, every kv head).  src == dst is a no-op.  A pair with an id outside
 *   [0, num_blocks) is skipped and sets PKV_DEVFLAG_BAD_BLOCK_ID.  If a dst is also a src,
 *   or two pairs share a dst, the result for those blocks is unspecified.
 *   num_pairs == 0 is a no-op returning PKV_OK.  The pool description is validated as for
 *   the append (PKV_ERR_INVALID_ARG before any launch); block_pairs must be 8-byte aligned.
 *   Asynchronous on stream, like every call here.
 */
pkv_status pkv_copy_blocks(const pkv_cache_desc* cache, const int64_t* block_pairs,
                           int64_t num_pairs, pkv_stream_t stream);

/*
 * Bytes of device workspace that pkv_paged_decode_attention needs for these sizes on the
 * current device (0 if the call needs none, i.e. when no sequence is split).  The workspace
 * holds per-partition partial results (running max, running sum, unnormalised output) of
 * the context split.  It needs no initialisation: every value a call reads was written by
 * the same call.  A workspace may not be used by two calls that can run at the same time.
 * Returns 0 and sets pkv_last_error() for invalid sizes.
 */
size_t pkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_context_len);

/* Context partition length (tokens, a multiple of 16) the decode uses for these sizes on
 * the current device; a sequence of n tokens is split into ceil(n / partition) parts. */
int32_t pkv_decode_partition_tokens(int32_t batch, int32_t num_kv_heads, int32_t max_context_len);

/*
 * Paged decode attention (section 3 definition, section 5 call shape, GQA of section 2).
 *   q: [batch][num_q_heads][head_dim] bf16, 16-byte aligned.
 *   block_tables: [batch][max_blocks_per_seq] int32 physical block ids, row-major.  Only
 *     the first ceil(context_lens[b] / 16) entries of row b are read.
 *   context_lens: [batch] int32, the number of cached tokens of each sequence (including
 *     a token appended this step).  0 gives an all-zero output row.
 *   max_context_len: an upper bound on every context_lens[b]; it sizes the launch.
 *   softmax_scale: multiplies q.k before the softmax (1/sqrt(head_dim) in section 3).
 *   out: [batch][num_q_heads][head_dim], bf16 (round to nearest even) or fp32.
 *   Query head hq reads kv head hq / (num_q_heads / num_kv_heads); num_q_heads must be a
 *   multiple of num_kv_heads with a quotient in {1, 2, 4, 8}.
 *   For each (b, hq), with n = context_lens[b]:
 *     out[b][hq] = sum_t softmax_t(scale * q[b][hq] . K_t) V_t,  t = 0 .. n-1,
 *   K_t/V_t the cached rows of kv head hq/G at position t (decoded times its scale for
 *   E4M3).  The result is deterministic: it depends only on the values, the lengths and
 *   the partition length, not on physical block ids, batch order or timing.
 *   Arithmetic: the per-block products run on the tensor cores with fp32 accumulation; K
 *   and V enter as stored (bf16, or E4M3 expanded exactly to fp16); q enters as bf16, or
 *   for E4M3 pools times a per-head power of two rounded to fp16 (relative error at most
 *   2^-11); the softmax weights enter as a 16-bit hi + lo pair.  While the environment
 *   variable PKV_DECODE_CUDA_CORES is "1" (read at each call), every product runs in fp32
 *   on the CUDA cores instead.  PKV_SPLIT_TOKENS (a positive multiple of 16, read at each
 *   call and by pkv_decode_workspace_size) fixes the partition length (tuning; the
 *   workspace size follows it).
 *   workspace: device memory of at least pkv_decode_workspace_size(...) bytes, 256-byte
 *   aligned, any contents; may be NULL when the required size is 0.
 */
pkv_status pkv_paged_decode_attention(const pkv_cache_desc* cache, const void* q,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t batch,
                                      int32_t num_q_heads, int32_t max_context_len,
                                      float softmax_scale, void* out, pkv_out_dtype out_dtype,
                                      void* workspace, size_t workspace_bytes,
                                      pkv_stream_t stream);

/*
 * One decode step in one launch: the append of pkv_paged_kv_append and the attention of
 * pkv_paged_decode_attention, for the shape of a decode step -- one new token per sequence,
 * token b being sequence b's token at position context_lens[b] - 1 (section 1: each step
 * computes K, V of the new token only, appends them, and attends over the cache that now
 * holds it; section 4 worked example: token 1025 goes to the next slot of the sequence's
 * last block).
 *   k, v: [batch][num_kv_heads][head_dim] bf16, 16-byte aligned: the new token of each
 *     sequence.  slot_mapping: [batch] int64, 8-byte aligned: the slot of that token, which
 *     must be the slot of position context_lens[b] - 1 in row b of block_tables; < 0: the
 *     sequence appends nothing this step (its attention still runs over the pool as it is).
 *   Everything else as for pkv_paged_decode_attention.
 *   Result: the pool and out are bit for bit those of pkv_paged_kv_append(cache, k, v,
 *   slot_mapping, batch) followed by pkv_paged_decode_attention(...) on the same stream.
 *   The tensor-core form stores each new token from the CTA that reads the sequence's last
 *   block and writes it into that CTA's copy of the block, so no separate launch and no
 *   re-read is needed.  A slot that is not position context_lens[b] - 1 of the table (or is
 *   outside the pool) sets PKV_DEVFLAG_BAD_SLOT; an in-pool one is stored, but the decode
 *   then reads that block as the pool held it before this call.  A sequence with
 *   context_lens[b] == 0 appends nothing.  With PKV_DECODE_CUDA_CORES=1 the two calls run
 *   one after the other.
 */
pkv_status pkv_paged_append_decode(const pkv_cache_desc* cache, const void* k, const void* v,
                                   const int64_t* slot_mapping, const void* q, const int32_t* block_tables,
                                   int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                                   int32_t num_q_heads, int32_t max_context_len, float softmax_scale, void* out,
                                   pkv_out_dtype out_dtype, void* workspace, size_t workspace_bytes,
                                   pkv_stream_t stream);

/*
 * Decode attention without a caller-provided workspace.  (The pages describe no such
 * call; it serves callers that cannot allocate device memory when they run a decode step:
 * an allocator that has reserved all device memory for itself, a serving loop that
 * forbids allocation after start-up, or a C caller with no allocator at hand.)
 *   Arguments, results and errors are those of pkv_paged_decode_attention; the workspace
 *   is a fixed 32 MiB array inside the library, one per device that loads it.
 *   Calls whose workspace would exceed 32 MiB (pkv_decode_workspace_size) are rejected with
 *   PKV_ERR_WORKSPACE before anything is enqueued.
 *   The first call on a device looks up that device's copy of the array (with the device
 *   current); make that first call before any stream capture.
 *   All calls on a device share the one array, and it keeps what the last call left: it is
 *   never cleared, and needs not be, since every value a call reads from it was written by
 *   that same call.  Two calls whose work can overlap on the GPU (different streams, or
 *   different host threads on one device) race on it.
 *   It allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
pkv_status pkv_paged_decode_attention_noalloc(const pkv_cache_desc* cache, const void* q,
                                              const int32_t* block_tables,
                                              int32_t max_blocks_per_seq,
                                              const int32_t* context_lens, int32_t batch,
                                              int32_t num_q_heads, int32_t max_context_len,
                                              float softmax_scale, void* out,
                                              pkv_out_dtype out_dtype, pkv_stream_t stream);

/*
 * Two-level (cascade) decode attention for sequences that share a prompt prefix.
 * (section 7, "Тот самый Cache Read": requests with the same prompt read the same cached
 * prefix blocks; section 3: attention over a split of the keys into parts is recovered
 * exactly from each part's running max, running sum and unnormalised output.)
 * The result for every (b, hq) is the decode attention of q[b][hq] over the concatenation
 * (prefix blocks of sequence b, if any) then (the blocks of block_tables row b), exactly
 * as pkv_paged_decode_attention over that concatenated table computes it, up to fp32
 * rounding.  The prefix part is computed once per prefix for all its member sequences,
 * as a dense [members x G rows] x [prefix keys] contraction: on the fifth-generation tensor
 * cores (tcgen05 MMAs of 128 query rows, fp32 accumulation in tensor memory), or, for an
 * E4M3 pool whose groups hold at most 32 query rows (max_members x G <= 32), on mma.sync
 * tensor-core tiles of 16 rows that expand the codes straight into their operands; the
 * sequences' own blocks go through the decode kernel, and the prefix results are merged
 * with log-sum-exp weights by a merge kernel after the decode (so that no decode CTA waits
 * for the prefix pass; for bf16 pools the pass runs beside the decode).
 *   prefixes: see pkv_prefix_desc; may describe zero prefixes (then this is a plain decode).
 *   block_tables / context_lens: each sequence's blocks AFTER its prefix and their token
 *     count (its full table and length when it has no prefix); 0 is allowed when the
 *     prefix is the whole context.
 *   Other arguments as for pkv_paged_decode_attention; workspace of at least
 *   pkv_cascade_workspace_size(...) bytes (never 0 when prefixes exist), any contents.
 *   Arithmetic of the prefix part: bf16 pools multiply bf16 q and K, and the softmax
 *   weights enter the P V product as a bf16 hi + lo pair (about 16 significant bits);
 *   E4M3 pools expand the codes exactly to fp16, multiply fp16 q (q rounded to fp16, exact
 *   for |q| in 2^-14 .. 65504) and fp16 weights; the tcgen05 pass sums the rounded weights
 *   into the denominator, the mma.sync pass the fp32 weights before rounding (either way
 *   each weight's relative error is at most 2^-11).
 *   Tuning (environment, read at each call; results agree within the tolerances above):
 *   PKV_PREFIX_SPLIT_BLOCKS (>= 4) fixes the prefix blocks per split of the prefix pass,
 *   PKV_PREFIX_CTAS_PER_SM (1 up to the pass's CTAs that fit an SM) the prefix-pass CTAs an SM
 *   is planned for, and
 *   PKV_CASCADE_DEFER (0 or 1) whether the prefix records are merged in the decode kernel (0)
 *   or by the merge kernel after it (1), and PKV_PREFIX_PASS ("tc" or "mma") which prefix
 *   pass runs where both apply; PKV_SPLIT_TOKENS applies as for the plain decode.
 */
typedef struct {
  const int32_t* prefix_tables;  /* [num_prefixes][max_prefix_blocks] physical block ids */
  int32_t max_prefix_blocks;
  const int32_t* prefix_lens;    /* [num_prefixes] tokens, each a multiple of 16 (whole
                                    blocks are shared) and <= max_prefix_len */
  int32_t num_prefixes;
  const int32_t* member_indptr;  /* [num_prefixes + 1]: the members of prefix p are */
  const int32_t* member_seqs;    /* member_seqs[member_indptr[p] .. member_indptr[p+1]) */
  int32_t max_members;           /* upper bound on the members of one prefix */
  int32_t max_prefix_len;        /* upper bound on prefix_lens (tokens) */
  const int32_t* seq_prefix;     /* [batch]: p for a member of prefix p, else -1; every
                                    sequence belongs to at most one prefix and must appear
                                    in that prefix's member list */
} pkv_prefix_desc;

size_t pkv_cascade_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_context_len,
                                  int32_t num_prefixes, int32_t max_members,
                                  int32_t max_prefix_len);

pkv_status pkv_cascade_decode_attention(const pkv_cache_desc* cache, const void* q,
                                        const pkv_prefix_desc* prefixes,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* context_lens, int32_t batch,
                                        int32_t num_q_heads, int32_t max_context_len,
                                        float softmax_scale, void* out, pkv_out_dtype out_dtype,
                                        void* workspace, size_t workspace_bytes,
                                        pkv_stream_t stream);

/*
 * Checksum of the cached K and V of every (sequence, kv head), read through the block
 * tables.  (The pages describe no such call.  It checks a pool's contents, e.g. after a
 * block copy, and it is the decode's read pattern with nothing else: the same grid, TMA
 * loads and partition length, so its time is the practical ceiling of the decode's reads.)
 *   block_tables, max_blocks_per_seq, context_lens, batch, max_context_len: as for
 *     pkv_paged_decode_attention (only the first ceil(context_lens[b] / 16) ids of row b
 *     are read; out-of-range lengths are clamped and ids outside the pool read as zeros,
 *     both flagged in the device status word).
 *   checksums: device uint32 [batch][num_kv_heads][2], 4-byte aligned; entry [b][h][0]
 *     covers K, [b][h][1] V.  With n = context_lens[b] and x_t the XOR of the 32-bit
 *     little-endian words of row t of kv head h (head_dim elements as stored),
 *       checksum = XOR over t = 0 .. n-1 of rotl32(x_t, t mod 32).
 *   The call clears `checksums` on `stream` before it reads; batch == 0 is a no-op.
 */
pkv_status pkv_paged_kv_checksum(const pkv_cache_desc* cache, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                                 int32_t max_context_len, uint32_t* checksums, pkv_stream_t stream);

/*
 * Copy `bytes` bytes from src to dst with the SMs, in order with the work on `stream`.
 * (The pages describe no such call.  It moves a decode step's inputs from page-locked host
 * memory to the device and its output back: on GB300 a copy-engine transfer of a few
 * hundred KiB costs about 10 us, nearly all latency, where the SMs read or write page-locked
 * host memory directly over the host link in a few.)
 *   dst, src: device memory or page-locked host memory (cudaHostAlloc, cudaHostRegister,
 *     or a pinned tensor: the same pointer addresses it on the device); both 16-byte
 *     aligned; the two ranges must not overlap.
 *   bytes: a multiple of 16; 0 is a no-op.
 * The copy starts once the work queued on `stream` before it has completed, and lets the
 * next kernel's launch proceed meanwhile (programmatic dependent launch).  Errors: a NULL or
 * misaligned pointer, a size not a multiple of 16 or overlapping ranges give
 * PKV_ERR_INVALID_ARG before any CUDA call; so does a pointer to memory that is neither
 * device, page-locked host nor managed memory (checked with the runtime's pointer query).
 */
pkv_status pkv_stage_copy(void* dst, const void* src, size_t bytes, pkv_stream_t stream);

/*
 * Read and clear the device status word of the current device after the work queued on
 * `stream` so far has finished (this call synchronises `stream`).  *flags receives the
 * PKV_DEVFLAG_* bits (may be NULL).  Returns PKV_ERR_DEVICE_CHECK if any bit was set,
 * PKV_OK if none, PKV_ERR_CUDA if reading it failed.
 */
pkv_status pkv_check_device_status(pkv_stream_t stream, uint32_t* flags);

/* Static description of a status code. */
const char* pkv_status_string(pkv_status s);

/* Message of the last failed call on this thread ("" if none). */
const char* pkv_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int32_t pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
