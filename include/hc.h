/*
 * hc.h - C ABI of the GB300 (sm_103a) KV-cache wire codec with relative-RoPE fetch.
 *
 * The operations follow "HyperCache - Distributed KV-cache quantization and
 * relative RoPE reuse":
 *   - evict/encode: blocks are compressed before they leave the GPU's paged KV
 *     buffer ("Core Design", compression paragraph), to FP8 E4M3 for the wire
 *     or to grouped INT4 ("Example output", part B);
 *   - fetch/decode: a cached block reused at a new offset has every post-RoPE
 *     key pair rotated by delta-m = m_new - m_old, using the SO(2) identity
 *     R(m_new t) = R(delta-m t) R(m_old t) ("Core Design", relative RoPE
 *     paragraph), dequantized and rotated "on the fly" ("Example output",
 *     part B, live fetch), then placed in the paged buffer.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument documented as "device" must point to memory the
 *   current CUDA device can access; every call enqueues work on `stream`
 *   (a cudaStream_t; NULL = the legacy default stream) and returns without
 *   synchronizing.  The library allocates, frees and synchronizes nothing and
 *   keeps no mutable global state (only constants computed once per process);
 *   calls are thread-safe.
 * - Host-side argument errors return a negative hc_status synchronously and
 *   launch nothing.  A failed launch returns HC_ERR_CUDA.
 * - Data errors found on the device (a slot id outside [0, num_slots), a
 *   delta index outside [0, n_distinct), an n_valid outside [1, block_size])
 *   OR a bit (HC_DEVERR_*) into the caller's device int32 `err_flag` and skip
 *   that block; they never trap.  The library never clears `err_flag`: zero it
 *   before the call, read it after synchronizing.
 * - Keys and values must be finite.
 *
 * Paged buffer (one for K, one for V), per layer: `num_slots` slots, each
 * holding block_size tokens x n_kv_heads x d_head elements, token-major:
 *   element (layer l, slot s, token t, head h, channel c) is at
 *   base + l*layer_stride + s*slot_stride + (t*n_kv_heads + h)*d_head + c.
 *
 * Wire buffers, for a call over n_blocks blocks (kv = 0 is K, 1 is V):
 *   FP8 : codes  u8  [n_layers][n_blocks][2][n_kv_heads][block_size][d_head]
 *         scales f32 [n_layers][n_blocks][2][n_kv_heads]           (per block, head)
 *   FP8_ROWS: codes as FP8
 *         scales f16|f32 [n_layers][n_blocks][2][n_kv_heads][block_size] (per token row)
 *   INT4: codes  u8  [n_layers][n_blocks][2][n_kv_heads][block_size][d_head/2]
 *                    (channel 2k in the low nibble, 2k+1 in the high nibble,
 *                     4-bit two's complement, values -7..7)
 *         scales f16|f32 [n_layers][n_blocks][2][n_kv_heads][block_size][d_head/group]
 *   RAW : values in the paged dtype, [n_layers][n_blocks][2][n_kv_heads][block_size][d_head]
 *         (unquantized; no scales).
 * Padding rows (token t >= n_valid[j]) are encoded as code 0 (INT4 and
 * FP8_ROWS scale 0).
 */
#ifndef HC_H_
#define HC_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HC_API_VERSION 3

typedef enum hc_status {
  HC_OK = 0,
  HC_ERR_INVALID_ARG = -1, /* a null pointer, bad size, bad alignment or unknown enum */
  HC_ERR_UNSUPPORTED = -2, /* valid but not built: d_head, block_size, group, dtype combination */
  HC_ERR_CUDA = -3         /* the CUDA runtime reported an error at launch */
} hc_status;

typedef enum hc_dtype { HC_F32 = 0, HC_F16 = 1, HC_BF16 = 2 } hc_dtype;

/* Which channels form a rotation pair: (2i, 2i+1), or (i, i + d_head/2). */
typedef enum hc_pairing { HC_PAIR_INTERLEAVED = 0, HC_PAIR_HALF_SPLIT = 1 } hc_pairing;

typedef enum hc_wire {
  HC_WIRE_FP8 = 0,     /* E4M3, one fp32 scale per (layer, block, kv, head) */
  HC_WIRE_INT4 = 1,    /* grouped INT4 */
  HC_WIRE_RAW = 2,     /* unquantized */
  HC_WIRE_FP8_ROWS = 3 /* E4M3, one scale per (layer, block, kv, head, token) row */
} hc_wire;

/* Bits ORed into *err_flag by the device. */
#define HC_DEVERR_SLOT 1   /* src_slots[j] or dst_slots[j] outside [0, num_slots) */
#define HC_DEVERR_DELTA 2  /* delta_idx[j] outside [0, n_distinct) */
#define HC_DEVERR_NVALID 4 /* n_valid[j] outside [1, block_size] */

/* Shape and strides of one paged buffer pair (K and V share it).
 * Supported: d_head in {64, 128}; block_size in {16, 32, 64, 128};
 * n_kv_heads >= 1; n_layers >= 1; num_slots >= 1.
 * slot_stride >= block_size*n_kv_heads*d_head; layer_stride may be any value
 * (0 is fine for n_layers == 1); both in elements, and both times the element
 * size must be multiples of 16 bytes.  The K and V base pointers must be
 * 16-byte aligned. */
typedef struct hc_paged_desc {
  int32_t n_layers;
  int32_t n_kv_heads;
  int32_t d_head;
  int32_t block_size;
  int32_t num_slots;
  int32_t dtype; /* hc_dtype */
  int64_t slot_stride;  /* elements between slot s and s+1 of one layer */
  int64_t layer_stride; /* elements between layer l and l+1 */
} hc_paged_desc;

/* hc_encode_fp8: gather blocks src_slots[0..n_blocks) of every layer from the
 * paged K and V buffers and quantize each (layer, block, kv, head) slab of
 * block_size x d_head elements to FP8 E4M3 with one fp32 scale:
 *   amax = max |x| over the slab's valid tokens,  s = fp32(amax / 448),
 *   code = E4M3(fp32(x / s)), round to nearest even, saturating at +-448,
 *   sign kept (so -0 encodes as 0x80).  A slab with s == 0 gets all-zero codes.
 * [HyperCache page, "Core Design" compression paragraph; "Example output"
 *  part B, "FP8 (E4M3) Wire Quantization".]
 *
 *   paged_k, paged_v : device, read-only, layout per `desc` (dtype f32/f16/bf16)
 *   desc             : host pointer, read during the call only
 *   src_slots        : device int32 [n_blocks], slot of block j (same in all layers)
 *   n_valid          : device int32 [n_blocks] valid tokens of block j, or NULL (all full)
 *   n_blocks         : >= 0; 0 launches nothing
 *   codes            : device u8, FP8 wire layout above, 16-byte aligned, written in full
 *   scales           : device f32, FP8 scale layout above, written in full
 *   err_flag         : device int32, HC_DEVERR_* bits ORed in; blocks with a bad
 *                      src_slots[j] or n_valid[j] are skipped (their wire bytes
 *                      are left as they were)
 * Returns HC_OK, HC_ERR_INVALID_ARG, HC_ERR_UNSUPPORTED or HC_ERR_CUDA. */
int hc_encode_fp8(const void* paged_k, const void* paged_v, const hc_paged_desc* desc,
                  const int32_t* src_slots, const int32_t* n_valid, int32_t n_blocks,
                  uint8_t* codes, float* scales, int32_t* err_flag, void* stream);

/* hc_encode_fp8_crc: hc_encode_fp8, and in the same pass the CRC-32 of every
 * slab: crc[((l*n_blocks + j)*2 + kv)*n_kv_heads + h] = the CRC-32 (as
 * hc_crc32 defines it) of the slab's block_size*d_head code bytes followed by
 * the 4 bytes of its fp32 scale - hc_crc32(codes, B*d, B*d, scales, 4, 4,
 * n_slabs).  For fp16/bf16 sources the CRC is folded into the encode as the
 * codes are produced, and the slabs of a skipped block (a bad src_slots[j] or
 * n_valid[j]) get no CRC: their crc entries are left as they were.  For fp32
 * sources the call runs the CRC kernel over every slab after the encode, so a
 * skipped block's entries hold the CRC of its wire bytes as they stand (the
 * bytes it had before the call).
 * [HyperCache page, "Example output" part B: blocks stored with CRC32.]
 *
 *   crc : device u32 [n_layers][n_blocks][2][n_kv_heads], 4-byte aligned
 * Other arguments as for hc_encode_fp8. */
int hc_encode_fp8_crc(const void* paged_k, const void* paged_v, const hc_paged_desc* desc,
                      const int32_t* src_slots, const int32_t* n_valid, int32_t n_blocks,
                      uint8_t* codes, float* scales, uint32_t* crc, int32_t* err_flag,
                      void* stream);

/* hc_encode_int4: as hc_encode_fp8, but symmetric INT4 with one scale per
 * (layer, block, kv, head, token, group of `group` consecutive channels):
 *   s32 = fp32(amax / 7);  s = fp16_rne(s32) if scale_dtype == HC_F16, else s32;
 *   code = clamp(round_half_even(fp32(x / s)), -7, 7) using the stored s.
 * A group with s == 0 gets all-zero codes; padding rows get scale 0.
 * [HyperCache page, "Example output" part B, "INT4 (Grouped) L3 Disk".]
 *
 *   group       : 32, 64 or 128, and <= d_head
 *   scale_dtype : HC_F16 or HC_F32
 *   codes       : device u8, INT4 wire layout above, 16-byte aligned
 *   scales      : device f16 or f32, INT4 scale layout above, aligned to its element
 * Other arguments as for hc_encode_fp8. */
int hc_encode_int4(const void* paged_k, const void* paged_v, const hc_paged_desc* desc,
                   const int32_t* src_slots, const int32_t* n_valid, int32_t n_blocks,
                   int32_t group, int32_t scale_dtype, uint8_t* codes, void* scales,
                   int32_t* err_flag, void* stream);

/* hc_encode_fp8_rows: as hc_encode_fp8, but one scale per (layer, block, kv,
 * head, token) row of d_head channels - the granularity whose sizes match the
 * FP8 frame the page prints (131,072 fp16 values -> 131,072 code bytes +
 * 1,024 fp16 scales = 133,120 bytes, 1.97x):
 *   amax = max |x| over the row,  s32 = fp32(amax / 448),
 *   s = fp16_rne(s32) if scale_dtype == HC_F16, else s32,
 *   code = E4M3(fp32(x / s)) with the stored s, nearest even, saturating at
 *   +-448, sign kept.  A row with s == 0 gets all-zero codes; an fp16 scale
 *   that overflows (amax above about 2.9e7) is stored as +inf and gives the
 *   codes of x / inf = +-0.  Padding rows get scale 0 and codes 0.
 * [HyperCache page, "Example output" part B, "FP8 (E4M3) Wire Quantization"
 *  and "Live TCP Socket Fetch" frame size.]
 *
 *   scale_dtype : HC_F16 or HC_F32
 *   codes       : device u8, FP8_ROWS code layout above, 16-byte aligned
 *   scales      : device f16 or f32, FP8_ROWS scale layout above, aligned to its element
 * Other arguments as for hc_encode_fp8. */
int hc_encode_fp8_rows(const void* paged_k, const void* paged_v, const hc_paged_desc* desc,
                       const int32_t* src_slots, const int32_t* n_valid, int32_t n_blocks,
                       int32_t scale_dtype, uint8_t* codes, void* scales, int32_t* err_flag,
                       void* stream);

/* hc_build_delta_sincos: the rotation table of the fetch.  For each distinct
 * delta-m value n and pair i < d_head/2:
 *   theta_i = inv_freq[i] if inv_freq != NULL, else rope_base^(-2i/d_head);
 *   table[n][i] = ( fp32(cos(delta_m[n] * theta_i)), fp32(sin(delta_m[n] * theta_i)) )
 * with theta, the angle and cos/sin in fp64, each entry rounded once to fp32.
 * [HyperCache page, "Core Design" relative RoPE paragraph; theta_i as in the
 *  "Module 13: KV handoff" code listing, rope_cache.]
 *
 *   delta_m    : device int32 [n_distinct]
 *   n_distinct : >= 0; 0 launches nothing
 *   d_head     : even, 2..256
 *   rope_base  : > 0 (ignored when inv_freq is given)
 *   inv_freq   : device f64 [d_head/2] or NULL
 *   table      : device f32 [n_distinct][d_head/2][2] (cos, sin), 16-byte aligned
 */
int hc_build_delta_sincos(const int32_t* delta_m, int32_t n_distinct, int32_t d_head,
                          double rope_base, const double* inv_freq, float* table,
                          void* stream);

/* hc_fetch_rotate_scatter: for every layer and block j < n_blocks, decode the
 * wire slab (x = code_value * scale in fp32; RAW: the stored value), rotate
 * each K pair (x1, x2) by (c, s) = table[delta_idx[j]][i]:
 *   y1 = x1*c - x2*s,  y2 = x1*s + x2*c      (fp32; V is not rotated)
 * round to the paged dtype (nearest even) and write the valid token rows
 * t < n_valid[j] of K and V to slot dst_slots[j].  Nothing else is written.
 * [HyperCache page, "Core Design" relative RoPE paragraph; "Example output"
 *  part B, "Live TCP Socket Fetch + On-The-Fly RoPE".]
 *
 *   wire        : hc_wire (FP8, INT4, RAW or FP8_ROWS)
 *   codes       : device, wire layout above (RAW: paged dtype), 16-byte aligned
 *   scales      : device, wire scale layout above (RAW: ignored, may be NULL)
 *   group       : INT4 group size (32, 64, 128, <= d_head); ignored otherwise
 *   scale_dtype : INT4 and FP8_ROWS: HC_F16 or HC_F32; ignored otherwise
 *   table       : device f32 [n_distinct][d_head/2][2] from hc_build_delta_sincos,
 *                 16-byte aligned
 *   delta_idx   : device int32 [n_blocks], row of `table` for block j
 *   n_distinct  : rows in `table`, >= 1 when n_blocks > 0
 *   pairing     : hc_pairing
 *   dst_slots   : device int32 [n_blocks], destination slot of block j (same in
 *                 every layer).  Must be distinct (precondition, not checked).
 *   n_valid     : device int32 [n_blocks] or NULL (all full)
 *   paged_k, paged_v : device, written, layout per `desc`
 *   err_flag    : device int32; blocks with a bad slot, delta index or n_valid
 *                 are skipped and flagged
 */
int hc_fetch_rotate_scatter(int32_t wire, const void* codes, const void* scales, int32_t group,
                            int32_t scale_dtype, const float* table, const int32_t* delta_idx,
                            int32_t n_distinct, int32_t pairing, const int32_t* dst_slots,
                            const int32_t* n_valid, int32_t n_blocks, void* paged_k,
                            void* paged_v, const hc_paged_desc* desc, int32_t* err_flag,
                            void* stream);

/* hc_crc32: CRC-32 of encoded units, for tamper detection of stored or sent
 * blocks.  Unit u < n_units is the byte string
 *   a[u*a_stride .. u*a_stride + a_bytes) followed by b[u*b_stride .. u*b_stride + b_bytes)
 * (for instance one (layer, block)'s codes followed by its scales), and
 * crc[u] is its CRC-32/ISO-HDLC, the CRC of zlib and PNG: polynomial
 * 0x04C11DB7 processed bit-reflected, initial register 0xFFFFFFFF, final
 * xor 0xFFFFFFFF (check value 0xCBF43926 for the ASCII "123456789").
 * [HyperCache page, "Example output" part B, "INT4 (Grouped) L3 Disk
 *  (.hckv + CRC32)", and the CRC32 tamper-detection tests it lists.]
 *
 *   a        : device, 16-byte aligned; a_stride a multiple of 16; a_bytes >= 0
 *   b        : device, any alignment, or NULL when b_bytes == 0.  b (and the
 *              last a_bytes % 16 bytes of a) is read byte by byte by one warp
 *              per unit: meant for a short trailer such as the scales; the
 *              16-byte words of a are read at full speed
 *   n_units  : >= 0; 0 launches nothing
 *   crc      : device u32 [n_units], written in full.  When there are few,
 *              large units (each is then cut into chunks across warps), the
 *              call first zeroes crc[] on `stream` and the chunks' terms are
 *              xor-ed into it; a concurrent reader of crc[] sees partial
 *              values until the call's work completes.
 * Returns HC_OK, HC_ERR_INVALID_ARG or HC_ERR_CUDA. */
int hc_crc32(const void* a, int64_t a_bytes, int64_t a_stride, const void* b, int64_t b_bytes,
             int64_t b_stride, int32_t n_units, uint32_t* crc, void* stream);

/* hc_drift_select: the tokens to recompute after cached chunks are reordered.
 * Layer-0 K/V depends only on the token embeddings, so the rotated layer-0 KV
 * is exact; the tokens whose layer-0 hidden state drifted most are recomputed
 * through the deeper layers.  For each sequence s < n_seq and token t:
 *   drift[s][t] = sqrt( sum_c (h_fresh[s][t][c] - h_cached[s][t][c])^2 )
 * (differences, squares and the sum in fp32; the sum's order is the
 * library's), and selected[s][0..k) = the k tokens with the largest drift,
 * ties to the lower index, in ascending order.  The caller picks k, or
 * passes k <= 0 for the page's share, hc_selection_size(n_tokens).
 * [HyperCache page, "Core Design", selective recomputation: about 15% of the
 *  tokens, those whose layer-0 hidden state moved furthest, are recomputed,
 *  as in CacheBlend.]
 *
 *   h_cached, h_fresh : device, dtype f32/f16/bf16, 16-byte aligned; element
 *                       (s, t, c) at base + s*seq_stride + t*token_stride + c
 *   n_seq        : >= 0; 0 launches nothing.  n_seq * n_tokens < 2^31
 *   n_tokens     : >= 1
 *   hidden       : a multiple of 8, >= 8
 *   token_stride : >= hidden; seq_stride >= n_tokens * token_stride when
 *                  n_seq > 1; both in elements, times the element size a
 *                  multiple of 16 bytes
 *   k            : 1 <= k <= n_tokens, or <= 0 for hc_selection_size(n_tokens)
 *   drift        : device f32 [n_seq][n_tokens], written in full
 *   selected     : device int32 [n_seq][k] (k after the default is applied),
 *                  written in full
 * Hidden states must be finite.  Returns HC_OK, HC_ERR_INVALID_ARG or HC_ERR_CUDA. */
int hc_drift_select(const void* h_cached, const void* h_fresh, int32_t dtype, int32_t n_seq,
                    int32_t n_tokens, int32_t hidden, int64_t token_stride, int64_t seq_stride,
                    int32_t k, float* drift, int32_t* selected, void* stream);

/* hc_selection_size: the number of tokens per sequence that hc_drift_select
 * recomputes by default: ceil(15% of n_tokens), computed exactly in integers
 * as ceil(3 * n_tokens / 20); 1 or more for n_tokens >= 1, 0 for
 * n_tokens <= 0.  A host function (nothing runs on the GPU).
 * [HyperCache page, "Core Design", selective recomputation: about 15% of the
 *  tokens are recomputed.] */
int32_t hc_selection_size(int32_t n_tokens);

/* Block digests for cache lookup (host functions: every pointer is a host
 * pointer; nothing runs on the GPU).  Two deterministic 128-bit BLAKE2b
 * digests per block of block_size tokens, keyed by a per-tenant secret
 * derived with HMAC-SHA256, with a public namespace for shared prefixes.
 * [HyperCache page, "Core Design", item 1 "Dual-Mode Block Hashing".]
 *
 * hc_tenant_key: key_out[0..32) = HMAC-SHA256(master, "hc-tenant:" || tenant),
 *   or HMAC-SHA256(master, "hc-public") when tenant is NULL or "" (the public
 *   namespace).  master_len >= 0; tenant at most 4096 bytes. */
int hc_tenant_key(const uint8_t* master, int32_t master_len, const char* tenant,
                  uint8_t* key_out);

/* hc_block_digests: blocks j < ceil(n_tokens / block_size) of `tokens`
 * (block j = tokens [j*block_size, (j+1)*block_size), the last one may be
 * short), each token as 4 little-endian bytes:
 *   content_digests[j] = BLAKE2b-128(key; tokens of block j)
 *   prefix_digests[j]  = BLAKE2b-128(key; prefix_digests[j-1] || tokens of block j)
 * (prefix_digests[-1] is empty, so block 0's two digests are equal).  The
 * content digest names a chunk wherever it sits (reuse at a new offset with
 * the relative rotation); the prefix digest names it with everything before
 * it (exact causal reuse).  key_len 1..64 (a tenant key is 32 bytes); the
 * outputs hold 16 bytes per block.  BLAKE2b per RFC 7693, SHA-256 per
 * FIPS 180-4, HMAC per RFC 2104. */
int hc_block_digests(const int32_t* tokens, int64_t n_tokens, int32_t block_size,
                     const uint8_t* key, int32_t key_len, uint8_t* prefix_digests,
                     uint8_t* content_digests);

/* Human-readable name of an hc_status value (static string, never NULL). */
const char* hc_status_string(int32_t status);

/* Text of the last CUDA error seen by a call on this host thread ("" if none). */
const char* hc_last_cuda_error(void);

/* HC_API_VERSION of the loaded library. */
int32_t hc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HC_H_ */
