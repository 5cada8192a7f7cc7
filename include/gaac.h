/*
 * gaac.h — C ABI of the GAAC compressed-KV decode-attention library (GB300, sm_103a).
 *
 * Method: "GAAC: Lossless KV Compression for Bandwidth-Efficient LLM Inference on
 * Personal Devices" (Guo, George, Joshi).  The cache keeps each BF16 value's sign
 * and mantissa verbatim and codes its exponent as a calibrated per-channel base
 * plus a 3-bit or 4-bit offset, or raw, chosen per group of eight (section 3.1);
 * 64-token blocks are packed into fixed-capacity slots, oversized blocks and the
 * open tail stay BF16 (section 3.3, Figure 3); attention rebuilds tiles on the fly
 * instead of decompressing the cache (section 3.2).
 *
 * Conventions shared by every entry point
 *  - All array arguments are DEVICE pointers owned by the caller, except where a
 *    comment says host.  The library allocates no memory.
 *  - Calls enqueue work on `stream` and return at once.  The return value reports
 *    argument errors found on the host (GAAC_EINVAL) and launch failures
 *    (GAAC_ECUDA); nothing is enqueued when it is not GAAC_OK.
 *  - Errors found by kernels are written to `*d_status` (device int32, may be
 *    NULL): the first nonzero code wins (atomic compare-and-swap from 0).  Kernels
 *    never trap and never wait without a bound.  Read it after synchronising.
 *  - BF16 values are passed as their uint16_t bit patterns.
 *  - head_dim is 128 and the block is 64 tokens (format v3 below).
 *
 * Tile format v3 (identical in the CUDA library and in the test oracle):
 *  tile        64 tokens x 128 channels of one (layer, sequence, block, kv-head, K|V)
 *  order       K tiles token-major  (element (t,c) at s = t*128 + c);
 *              V tiles in tensor-core operand order:
 *                s = 1024*(2*(t/16) + c/64) + 32*(4*(c%8) + (t%8)/2) + 8*((c/16)%4)
 *                    + (c%16)/8 + 2*(t%2) + 4*((t%16)/8)
 *              (32-element unit 32*(2w+h) + 4g + q holds channels 16m+g and
 *              16m+g+8, m = 4h..4h+3, at tokens 16w + 2q + {0,1,8,9})
 *  group       8 consecutive elements in that order (G = s/8)
 *  slot image  GAAC_SLOT_BYTES bytes:
 *               [0,8192)      byte s: mantissa of element s in bits 0-6; bit 7 is
 *                             the sign of element 4*(s/4) + (s+3)%4 (the signs of
 *                             each aligned group of four rotated by one byte)
 *               [8192,11264)  3-bit codes: word k (0..2) of 32-element unit u at
 *                             8192 + 4*(k*256 + u); raw groups have code 0
 *               [11264,11520) 2-bit mode of group G at byte 11264 + G/4, bits 2*(G%4)
 *               [11520,11536) escape directory: 8 little-endian u16; entry w is
 *                             (4-bit groups in [0, 128*(w+1))) mod 512
 *                             + 512 * ((raw groups there) mod 128)
 *               [11536,12032) escape area, zero filled, capacity 496: one byte per
 *                             4-bit group (bit j = bit 3 of element j's offset), in
 *                             group order; then eight bytes per raw group (its
 *                             exponents), in group order
 *  raw tile    8192 BF16 words in the same storage order
 */
#ifndef GAAC_H
#define GAAC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GAAC_API __attribute__((visibility("default")))
#else
#define GAAC_API
#endif

#define GAAC_HEAD_DIM 128
#define GAAC_BLOCK 64
#define GAAC_TILE_ELEMS 8192
#define GAAC_SLOT_BYTES 12032
#define GAAC_ESC_CAPACITY 496
#define GAAC_RAW_TILE_BYTES 16384
#define GAAC_MAX_GQA 8 /* query heads per kv-head supported by decode attention */

/* Status codes (return values and *d_status). */
enum {
  GAAC_OK = 0,
  GAAC_EINVAL = 1,   /* bad argument (host) or bad base / length (device) */
  GAAC_EPOOL = 2,    /* raw-tile free list or slot index out of range */
  GAAC_EFORMAT = 3,  /* reserved mode tag, bad table entry, escape past its length */
  GAAC_ECUDA = 4,    /* a CUDA launch failed */
  GAAC_ETIMEOUT = 5  /* a bounded wait inside a kernel gave up (data of that launch invalid) */
};

/* Flags of gaac_encode_blocks_ex and gaac_append_ex. */
#define GAAC_OPEN_COMPRESSED 1u /* keep the open (last, partial) block compressed in its slot */

/* Table entry modes. */
enum { GAAC_MODE_SLOT = 0, GAAC_MODE_RAW = 1, GAAC_MODE_NONE = 255 };

/* Slot-table entry (section 3.3: a table keeps, per block, whether it is
 * compressed or raw and where it lives).  One per (sequence, block, kv-head, K|V) of a layer, laid out
 * table[batch][max_blocks][n_kv_heads][2]  (last index 0 = K, 1 = V). */
typedef struct gaac_entry {
  uint32_t index;   /* slot index (mode SLOT) or raw-tile index (mode RAW) */
  uint16_t esc_len; /* bytes of the escape area used: 4-bit bytes + 8 per raw group (mode SLOT) */
  uint8_t mode;     /* GAAC_MODE_* */
  uint8_t n_tok;    /* tokens held: 64 for a sealed block, fewer for the open tail */
} gaac_entry;

/* Storage of one layer's compressed cache (all device pointers). */
typedef struct gaac_pools {
  uint8_t* slot_pool;       /* [n_slots][GAAC_SLOT_BYTES] */
  int64_t n_slots;
  uint16_t* raw_pool;       /* [n_raw][GAAC_TILE_ELEMS] */
  int64_t n_raw;
  const uint32_t* raw_free; /* free raw-tile indices, popped at raw_free[*raw_cursor]; NULL = identity list */
  int64_t n_raw_free;       /* length of the free list (identity list: n_raw) */
  uint32_t* raw_cursor;     /* device counter of popped entries */
} gaac_pools;

/* Optional encoder counters (device, accumulated with atomics). */
typedef struct gaac_stats {
  unsigned long long groups[4];     /* groups per mode tag 0..3 in encoded slots */
  unsigned long long escape_bytes;  /* sum of esc_len over encoded slots */
  unsigned long long slot_tiles;    /* tiles stored compressed */
  unsigned long long raw_tiles;     /* full tiles that fell back to BF16 */
  unsigned long long tail_tiles;    /* partial (open) tiles written as BF16 */
} gaac_stats;

/* Human-readable name of a status code (static string). */
GAAC_API const char* gaac_strerror(int status);

/* Library version of the tile format and of the ABI. */
GAAC_API int gaac_format_version(void);

/*
 * Calibration (section 3.1: each head-channel gets a window of 8 and a window
 * of 16 exponents, fixed from calibration data; section 4.7.1).  For each kv-head h and channel c, counts
 * the exponents of x[t*tok_stride + h*128 + c] over t < n_tok and picks
 *   base3[h*128+c] = argmax_{b in [0,248]} sum_{i<8}  count[b+i]
 *   base4[h*128+c] = argmax_{b in [0,240]} sum_{i<16} count[b+i]
 * (ties: smallest b).  Call once for K and once for V.
 * x: BF16 bits, tok_stride in elements (>= n_kv_heads*128).  1 <= n_tok <= 65535.
 */
GAAC_API int gaac_calibrate(const uint16_t* x, int64_t n_tok, int64_t tok_stride, int n_kv_heads, uint8_t* base3,
                   uint8_t* base4, int32_t* d_status, void* stream);

/*
 * Block encoder for prefill (section 3.3: at prefill the full blocks are
 * compressed and the partial last block is kept as BF16).  For every sequence b
 * with length seq_lens[b] and every kv-head and K|V:
 *  - each complete block is encoded into slot slot_ids[((b*max_blocks+blk)*H+h)*2+kv]
 *    (mode SLOT), or, if its escape stream exceeds GAAC_ESC_CAPACITY, copied as a
 *    raw tile popped from the raw free list (mode RAW; that slot stays unused);
 *  - the incomplete last block, if any, is copied into a raw tile popped from
 *    the free list (mode RAW, n_tok = tokens held, the rest zero);
 *  - table entries of blocks past the sequence are set to GAAC_MODE_NONE.
 * slot_ids may be NULL: every block is then stored as a raw tile (an
 * uncompressed BF16 cache in the same paged layout, read by the same attention
 * kernel; used as the uncompressed baseline).
 * k, v: BF16 bits, element (b, t, h, c) at b*seq_stride + t*tok_stride + h*128 + c.
 * base3/base4: [2][n_kv_heads][128] bytes (index 0 = K, 1 = V), 16-byte aligned.
 * k and v must be 16-byte aligned and both strides multiples of 8 elements
 * (a misaligned pointer or stride returns GAAC_EINVAL).
 * n_tok: tokens present per sequence in k and v.  Each seq_lens[b] must be
 * <= min(n_tok, max_blocks*64); otherwise GAAC_EINVAL goes to *d_status and the
 * sequence is left out (its entries become GAAC_MODE_NONE).
 */
GAAC_API int gaac_encode_blocks(const uint16_t* k, const uint16_t* v, int64_t seq_stride, int64_t tok_stride,
                       int64_t n_tok, const int32_t* seq_lens, int batch, int n_kv_heads, int max_blocks, const uint8_t* base3,
                       const uint8_t* base4, gaac_entry* table, const uint32_t* slot_ids, const gaac_pools* pools,
                       gaac_stats* stats, int32_t* d_status, void* stream);

/*
 * O(1) append of one decode token per sequence (section 3.3: decode tokens go
 * to a BF16 tail block, which is compressed a single time once it is full).
 * For each b, kv-head h, K|V: writes k_new/v_new[(b*n_kv_heads+h)*128 + c] at
 * position p = seq_lens[b] % 64 of block blk = seq_lens[b] / 64, whose tile must
 * be the open raw tail (a raw tile is popped from the free list when the block
 * has none yet; a new tail tile is cleared to zero first).  When the tile becomes full it is encoded into slot
 * slot_ids[((b*max_blocks+blk)*n_kv_heads+h)*2+kv] (same layout as for
 * gaac_encode_blocks); if it fits, the entry becomes SLOT and the raw tile is
 * handed to block blk+1 as its tail; if not, the block stays RAW.  slot_ids may be
 * NULL (a cache of raw tiles only, as gaac_encode_blocks writes with NULL): a full
 * tail then stays a RAW tile.  Finally seq_lens[b] += 1: with 2 * n_kv_heads <= 16
 * the CTAs of a sequence run as one thread-block cluster (one launch) and the
 * first advances the length once all have read it; with more kv-heads a second
 * small kernel on the same stream does it.
 * seq_lens[b] must be < max_blocks*64 (else GAAC_EINVAL in *d_status).
 * base3/base4 as for gaac_encode_blocks (16-byte aligned, else GAAC_EINVAL).
 */
GAAC_API int gaac_append(const uint16_t* k_new, const uint16_t* v_new, int32_t* seq_lens, int batch, int n_kv_heads,
                int max_blocks, const uint8_t* base3, const uint8_t* base4, gaac_entry* table,
                const uint32_t* slot_ids, const gaac_pools* pools, gaac_stats* stats, int32_t* d_status,
                void* stream);

/*
 * gaac_encode_blocks and gaac_append with flags.  flags = 0 is the plain call.
 *
 * GAAC_OPEN_COMPRESSED keeps the open block compressed (section 3.3 keeps the
 * last block open while decode tokens arrive; here it is stored in its slot
 * from its first token instead of as a BF16 tile).  The slot of an open block
 * holding n < 64 tokens is the image of its first n tokens in which the
 * elements of later tokens are absent: they take no part in their group's
 * mode, and their sign|mantissa bits (including the sign bit an element lends
 * to its neighbour's byte), codes, escape bits and raw exponent bytes are zero.
 * Directory entries and esc_len count the present groups' escapes.  Its table
 * entry is {slot, esc_len, GAAC_MODE_SLOT, n}.  With all 64 tokens present this
 * is the sealed encoding, so a block filled token by token ends in the same
 * bytes as one encoded at once.  Attention and decompression read open slots
 * like sealed ones (tokens past the sequence length are masked).
 *  - gaac_encode_blocks_ex: the incomplete last block of each sequence is
 *    encoded into slot_ids[...] of its block (slot_ids must not be NULL for
 *    the flag to apply); if its escape stream exceeds GAAC_ESC_CAPACITY, it is
 *    a raw tile as without the flag.  Open blocks are not counted in stats.
 *  - gaac_append_ex: a block that opens (position 0) takes slot
 *    slot_ids[((b*max_blocks+blk)*n_kv_heads+h)*2+kv] and holds the token as a
 *    one-token open image; a later token is added to the open slot by
 *    re-encoding its present tokens, writing only the 32-byte sign|mantissa
 *    rows and code words of the units that hold the new token (4 units for K,
 *    16 for V) and the tag plane, directory and escape area.  The work is
 *    bounded by one tile, whatever the sequence length.  If the escape stream
 *    of the open block outgrows the slot (it never shrinks as tokens arrive, so
 *    the full block would not fit either), its tokens so far move to a raw tile
 *    popped from the free list, and the block continues and seals as RAW.  A
 *    block whose entry is already a raw tail (from gaac_encode_blocks without
 *    the flag, or handed over by a raw tail that sealed into a slot) continues
 *    as gaac_append does.  A slot entry whose n_tok differs from seq_lens[b] %
 *    64, or an open image that fails the format checks, reports GAAC_EFORMAT and
 *    leaves the block untouched.
 * Unknown flag bits: GAAC_EINVAL.
 */
GAAC_API int gaac_encode_blocks_ex(const uint16_t* k, const uint16_t* v, int64_t seq_stride, int64_t tok_stride,
                          int64_t n_tok, const int32_t* seq_lens, int batch, int n_kv_heads, int max_blocks,
                          const uint8_t* base3, const uint8_t* base4, gaac_entry* table, const uint32_t* slot_ids,
                          const gaac_pools* pools, gaac_stats* stats, unsigned flags, int32_t* d_status,
                          void* stream);
GAAC_API int gaac_append_ex(const uint16_t* k_new, const uint16_t* v_new, int32_t* seq_lens, int batch,
                   int n_kv_heads, int max_blocks, const uint8_t* base3, const uint8_t* base4, gaac_entry* table,
                   const uint32_t* slot_ids, const gaac_pools* pools, gaac_stats* stats, unsigned flags,
                   int32_t* d_status, void* stream);

/*
 * Workspace bytes gaac_decode_attention needs for (batch, n_q_heads, n_splits).
 * n_splits = 0 asks for the automatic choice (max_blocks must then be given).
 */
GAAC_API size_t gaac_attention_workspace(int batch, int n_kv_heads, int max_blocks, int n_splits);

/*
 * Number of splits gaac_decode_attention uses for n_splits = 0.  A launch with
 * n_splits splits cuts every (sequence, kv-head) into chunks of
 * ceil(max_blocks / n_splits) blocks, one CTA each (one CTA per SM); a sequence
 * of nblk blocks uses max(1, ceil(nblk / chunk)) of them, so sequences of mixed
 * lengths give CTAs of equal work.  The automatic count minimises, for full
 * sequences, the number of waves of CTAs times (chunk + a CTA's fixed cost of
 * about 4 blocks).
 */
GAAC_API int gaac_attention_auto_splits(int batch, int n_kv_heads, int max_blocks);

/*
 * Fused split-K GQA decode attention over the compressed cache (section 3.2:
 * tiles are rebuilt inside the attention kernel, never decompressed to a full
 * cache, and compressed blocks and the raw tail feed one softmax).
 *   out[b][hq][c] = sum_{t < seq_lens[b]} softmax_t(scale * q[b][hq] . k[b][t][hk]) v[b][t][hk][c]
 * with hk = hq / (n_q_heads / n_kv_heads), in fp32 (0 for an empty sequence).
 * q: BF16 bits [batch][n_q_heads][128]; out: fp32 [batch][n_q_heads][128].
 * n_q_heads / n_kv_heads must be an integer <= GAAC_MAX_GQA.  scale: any finite
 * value (negative and zero included).  Every row whose logits scale * q . k_t are
 * fp32 numbers with |scale| * sum_c |q_c k_tc| below the largest fp32 value is
 * computed without overflow: the kernel subtracts each score's running maximum
 * before it applies the scale.
 * workspace: at least gaac_attention_workspace(...) bytes, 16-byte aligned.  It opens
 * with one counter per (sequence, kv-head) (u32, the block rounded up to 16 bytes)
 * that must be zero before the first call; every call leaves them at zero again,
 * whatever its split count, so one workspace serves calls with different counts.
 * The split partials follow the counters.
 * After a call that reported an error, zero the workspace before reusing it.
 * pools: only slot_pool, n_slots, raw_pool and n_raw are read; both pools must be
 * 16-byte aligned (tiles are fetched with bulk copies).  A table entry that is
 * neither a valid slot nor a valid raw tile reports GAAC_EFORMAT and its block
 * contributes nothing.
 */
GAAC_API int gaac_decode_attention(const uint16_t* q, int batch, int n_q_heads, int n_kv_heads, int max_blocks,
                          const int32_t* seq_lens, const gaac_entry* table, const gaac_pools* pools,
                          const uint8_t* base3, const uint8_t* base4, float scale, int n_splits, float* out,
                          void* workspace, size_t workspace_bytes, int32_t* d_status, void* stream);

/*
 * Decode attention over an uncompressed BF16 cache: the same kernel as
 * gaac_decode_attention (grid, staging ring, tensor-core QK^T and PV^T, online
 * softmax, split merge) specialised to raw tiles, with no decode path.  Every
 * table entry of a block below seq_lens must be a raw tile (mode GAAC_MODE_RAW,
 * 16 KiB of BF16 in the format's storage order in pools->raw_pool), as
 * gaac_encode_blocks writes them when slot_ids is NULL.  An entry of any other
 * mode reports GAAC_EFORMAT and its block contributes nothing.  It is the
 * uncompressed path the compressed cache is measured against: the GAAC page's
 * section 3.2 and Table 5 weigh the reads a compressed cache saves against the
 * reconstruction it adds.  Arguments, result, workspace and errors as
 * gaac_decode_attention, without bases; pools->slot_pool may be NULL.
 */
GAAC_API int gaac_decode_attention_bf16(const uint16_t* q, int batch, int n_q_heads, int n_kv_heads, int max_blocks,
                                        const int32_t* seq_lens, const gaac_entry* table, const gaac_pools* pools,
                                        float scale, int n_splits, float* out, void* workspace, size_t workspace_bytes,
                                        int32_t* d_status, void* stream);

/*
 * Decode attention for 256-channel heads (Appendix D: a 256-dimensional head is
 * stored as two 128-dimensional half-heads).  The cache holds 2 * n_kv_heads
 * half-heads: half-head 2h + j is channels [128 j, 128 j + 128) of kv-head h,
 * in the table ([batch][max_blocks][2 * n_kv_heads][2]) and in base3 / base4
 * ([2][2 * n_kv_heads][128]), i.e. the cache of a [batch][T][n_kv_heads][256]
 * K/V viewed as [batch][T][2 * n_kv_heads][128].  The attention runs over the
 * whole 256-channel head:
 *   out[b][hq][c] = sum_t softmax_t(scale * q[b][hq] . k[b][t][hk]) v[b][t][hk][c], c < 256
 * q: BF16 bits [batch][n_q_heads][256]; out: fp32 [batch][n_q_heads][256].
 * workspace: at least gaac_attention_workspace(batch, 2 * n_kv_heads, max_blocks,
 * n_splits) bytes; n_splits = 0 picks gaac_attention_auto_splits(batch,
 * 2 * n_kv_heads, max_blocks).  Everything else as gaac_decode_attention.
 */
GAAC_API int gaac_decode_attention_hd256(const uint16_t* q, int batch, int n_q_heads, int n_kv_heads, int max_blocks,
                                         const int32_t* seq_lens, const gaac_entry* table, const gaac_pools* pools,
                                         const uint8_t* base3, const uint8_t* base4, float scale, int n_splits,
                                         float* out, void* workspace, size_t workspace_bytes, int32_t* d_status,
                                         void* stream);

/*
 * Allocation-free decode attention.  The GAAC page has no counterpart; this is a
 * convenience of this library for callers that cannot allocate device memory
 * when they call it, such as a serving loop whose memory plan is fixed after
 * start-up, a plugin whose host owns all device allocations, or any code that
 * must not enter an allocator on the decode path.
 *
 * Same arguments, result and errors as gaac_decode_attention, without the
 * workspace: the split partials go to a scratch array of
 * GAAC_STATIC_SCRATCH_BYTES bytes that the library itself holds in device
 * memory on every GPU that loads it, until the process exits.  A call whose
 * partials would not fit (gaac_attention_workspace(batch, n_kv_heads,
 * max_blocks, n_splits) > GAAC_STATIC_SCRATCH_BYTES) returns GAAC_EINVAL and
 * enqueues nothing.  It calls no allocator (no cudaMalloc, no cudaFree).
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture.  Under CUDA's lazy module loading (the default) that
 *    first call may also be what loads the library's device code on the
 *    device, which reserves the array's 4 MiB there: a caller with a fixed
 *    memory plan makes the first call during start-up.
 *  - Every call shares the one array.  Calls whose kernels overlap on the GPU
 *    (other streams, other threads) race on it and give wrong results; issue
 *    them in one stream or order them.  The array keeps the last call's
 *    partials; each call first clears the merge counters it uses (a small
 *    memset on the same stream) and rewrites everything else it reads.
 */
#define GAAC_STATIC_SCRATCH_BYTES (4u << 20)
GAAC_API int gaac_decode_attention_noalloc(const uint16_t* q, int batch, int n_q_heads, int n_kv_heads,
                                           int max_blocks, const int32_t* seq_lens, const gaac_entry* table,
                                           const gaac_pools* pools, const uint8_t* base3, const uint8_t* base4,
                                           float scale, int n_splits, float* out, int32_t* d_status, void* stream);

/*
 * Decompress a layer's cache back to BF16 (section 4.3 compares block decode
 * latency; used for bit-exact checks).  Writes tokens t < seq_lens[b] of every
 * (b, h) to k_out/v_out at b*seq_stride + t*tok_stride + h*128 + c; n_tok is the
 * number of token rows the outputs hold (a longer sequence reports GAAC_EINVAL
 * and only its first n_tok tokens are written).
 * pools: slot_pool, n_slots, raw_pool, n_raw are read (16-byte aligned).  An
 * invalid entry reports GAAC_EFORMAT and its tokens are left untouched.
 */
GAAC_API int gaac_decompress(const gaac_entry* table, const int32_t* seq_lens, int batch, int n_kv_heads, int max_blocks,
                    const gaac_pools* pools, const uint8_t* base3, const uint8_t* base4, uint16_t* k_out,
                    uint16_t* v_out, int64_t seq_stride, int64_t tok_stride, int64_t n_tok, int32_t* d_status,
                    void* stream);

/*
 * FP8 variant of the codec (Appendix B, "Relation to FP8 KV": the same
 * exponent coding applied to a cache already quantised to FP8; lossless with
 * respect to the FP8 values).  GAAC-FP8 tile format v1:
 *  element   E4M3: sign(1) exponent(4) mantissa(3); E5M2: sign(1) exponent(5)
 *            mantissa(2); sm = sign << mantissa_bits | mantissa
 *  tile      64 x 128 FP8 bytes; storage order, groups, modes, codes, tags,
 *            directory and escape area as in format v3, the windows inside the
 *            format's 16 (E4M3: base4 is 0, no raw groups) or 32 exponents
 *  slot      E4M3 (7,936 B): [0,4096) sm nibbles (element s in byte s/2, low
 *            nibble for even s), [4096,7168) codes, [7168,7424) tags,
 *            [7424,7440) directory, [7440,7936) escape area;
 *            E5M2 (6,912 B): [0,3072) sm as 3-bit fields laid out like the
 *            code plane, [3072,6144) codes, [6144,6400) tags, [6400,6416)
 *            directory, [6416,6912) escape area
 */
enum { GAAC_FP8_E4M3 = 0, GAAC_FP8_E5M2 = 1 };

/* Slot bytes of an FP8 format (0 for an unknown format). */
GAAC_API int gaac_fp8_slot_bytes(int fmt);

/*
 * Windows of 8 and 16 exponents per (kv-head, channel) from FP8 calibration
 * data x[t*tok_stride + h*128 + c], t < n_tok: the windows holding the most
 * values, ties to the smallest base.  1 <= n_tok <= 65535.
 */
GAAC_API int gaac_fp8_calibrate(const uint8_t* x, int64_t n_tok, int64_t tok_stride, int n_kv_heads, int fmt,
                                uint8_t* base3, uint8_t* base4, int32_t* d_status, void* stream);

/*
 * Encodes n_tiles FP8 tiles tiles[i][64][128] (token-major; 16-byte aligned)
 * into slots[i][gaac_fp8_slot_bytes(fmt)] (16-byte aligned).  Tile i is K
 * (tile_kind[i] = 0) or V (1) and uses bases row tile_row[i] of base3 / base4
 * ([n_rows][128], 4-byte aligned).  esc_len[i] receives the escape-area length, or 0xFFFF when
 * the tile does not fit its slot (the caller keeps it as FP8; its slot is not
 * written).  stats may be NULL.  A bad kind or row sets GAAC_EINVAL in
 * *d_status and esc_len[i] = 0xFFFF.
 */
GAAC_API int gaac_fp8_encode_tiles(const uint8_t* tiles, int64_t n_tiles, int fmt, const uint8_t* tile_kind,
                                   const int32_t* tile_row, int n_rows, const uint8_t* base3, const uint8_t* base4,
                                   uint8_t* slots, uint16_t* esc_len, gaac_stats* stats, int32_t* d_status,
                                   void* stream);

/*
 * Decodes slot images back to FP8 tiles[i][64][128]; tiles whose esc_len is
 * 0xFFFF are skipped (not written).  A failed check reports GAAC_EFORMAT.
 */
GAAC_API int gaac_fp8_decompress_tiles(const uint8_t* slots, const uint16_t* esc_len, int64_t n_tiles, int fmt,
                                       const uint8_t* tile_kind, const int32_t* tile_row, int n_rows,
                                       const uint8_t* base3, const uint8_t* base4, uint8_t* tiles, int32_t* d_status,
                                       void* stream);

/*
 * Tile-batch codec, format v3 (the block encoder and decoder of the cache,
 * without the table): tiles[i][64][128] BF16 token-major, tile_kind[i] 0 = K,
 * 1 = V, tile_row[i] < n_rows selects the 128 bases base3/base4[row*128..].
 * gaac_encode_tiles writes slot image i at slots + i*GAAC_SLOT_BYTES and
 * esc_len[i], or esc_len[i] = 0xFFFF (slot untouched) when the escape stream
 * exceeds GAAC_ESC_CAPACITY; gaac_decode_tiles rebuilds tiles[i] from every
 * slot whose esc_len is not 0xFFFF.  tiles and slots 16-byte aligned, bases
 * 4-byte aligned.  A bad kind or row: GAAC_EINVAL in *d_status (esc_len 0xFFFF
 * on encode); a slot failing the format checks: GAAC_EFORMAT.
 */
GAAC_API int gaac_encode_tiles(const uint16_t* tiles, int64_t n_tiles, const uint8_t* tile_kind,
                               const int32_t* tile_row, int n_rows, const uint8_t* base3, const uint8_t* base4,
                               uint8_t* slots, uint16_t* esc_len, gaac_stats* stats, int32_t* d_status, void* stream);
GAAC_API int gaac_decode_tiles(const uint8_t* slots, const uint16_t* esc_len, int64_t n_tiles,
                               const uint8_t* tile_kind, const int32_t* tile_row, int n_rows, const uint8_t* base3,
                               const uint8_t* base4, uint16_t* tiles, int32_t* d_status, void* stream);

/*
 * Nested 2-bit-mode ablation format (section 4.7.2, Table 4: a 2-bit mode
 * nested inside the 3-bit one).  Not used by the cache; it measures the
 * ratio / decode-time trade of a variable code width.  Slot image of
 * GAAC_NESTED_SLOT_BYTES:
 *   [0,8192)      sign|mantissa plane, as format v3
 *   [8192,11264)  code stream: groups in group order; a 2-bit group takes 16
 *                 bits, a 3-bit or 4-bit group 24 (the 4-bit group's low three
 *                 offset bits), a raw group none; element j of a group at bit
 *                 (group start + j*width); bit b of the stream is bit b%8 of
 *                 byte b/8; zero past its end
 *   [11264,11520) tags, 2 bits per group: 0 3-bit, 1 4-bit, 2 raw, 3 2-bit
 *   [11520,11552) directory: 8 u32, entry w = 4-bit groups (mod 512) | raw
 *                 groups (mod 128) << 9 | code-stream bits << 16, each over
 *                 groups [0, 128(w+1))
 *   [11552,12048) escape area as format v3 (4-bit bytes, then raw exponents)
 * Mode rule: 2-bit if every offset from base2 is in [0,3], else format v3's.
 * gaac_nested_calibrate: base2[h*128+c] = the 4-exponent window holding the
 * most values of x[t*tok_stride + h*128 + c], t < n_tok, ties to the smallest
 * base.  The encode and decode calls follow gaac_encode_tiles and
 * gaac_decode_tiles (bases base2/base3/base4 [n_rows][128]).
 */
#define GAAC_NESTED_SLOT_BYTES 12048
GAAC_API int gaac_nested_calibrate(const uint16_t* x, int64_t n_tok, int64_t tok_stride, int n_kv_heads,
                                   uint8_t* base2, int32_t* d_status, void* stream);
GAAC_API int gaac_nested_encode_tiles(const uint16_t* tiles, int64_t n_tiles, const uint8_t* tile_kind,
                                      const int32_t* tile_row, int n_rows, const uint8_t* base2, const uint8_t* base3,
                                      const uint8_t* base4, uint8_t* slots, uint16_t* esc_len, int32_t* d_status,
                                      void* stream);
GAAC_API int gaac_nested_decode_tiles(const uint8_t* slots, const uint16_t* esc_len, int64_t n_tiles,
                                      const uint8_t* tile_kind, const int32_t* tile_row, int n_rows,
                                      const uint8_t* base2, const uint8_t* base3, const uint8_t* base4,
                                      uint16_t* tiles, int32_t* d_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GAAC_H */
