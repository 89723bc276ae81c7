// Internal declarations shared by the kernel translation units and the C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "hc.h"
#include "fastdiv.h"

namespace hc {

// One warp owns a "sub-slab": 16 consecutive token rows of one
// (layer, block, kv, head) slab.  A block of B tokens has B/16 sub-slabs, so a
// 256-thread CTA (8 warps) always holds whole slabs (B/16 divides 8).
constexpr int kThreads = 256;

// Fetch launch shape.  CTAS_PER_SM caps the grid at that many CTAs per SM
// (the CTAs then loop over units); the default large value gives one unit per
// CTA.  MIN_BLOCKS is the occupancy the register budget is sized for, and
// DOUBLE_BUFFER whether a warp loads its next unit while it computes the
// current one.  Measured on GB300, this write-heavy kernel is fastest with one
// unit per CTA, in CTAs of 4 warps (HC_FETCH_WARPS) at 7 per SM: 28 warps
// with 67 registers and no spills.  (The encoder picks its shape per call.)
#ifndef HC_FETCH_CTAS_PER_SM
#define HC_FETCH_CTAS_PER_SM (1 << 20)
#endif
#ifndef HC_FETCH_MIN_BLOCKS
#define HC_FETCH_MIN_BLOCKS 7
#endif
#ifndef HC_FETCH_DOUBLE_BUFFER
#define HC_FETCH_DOUBLE_BUFFER 0
#endif
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = 16;

// Flat work index -> (layer, block, kv, head, sub-slab).  A call has
// total = n_layers * n_blocks * 2 * H * wps sub-slabs (wps = block_size / 16),
// ordered ((layer * n_blocks + block) * 2H + kv * H + head) * wps + sub, so the
// wire slab index is (layer * n_blocks + block) * 2H + kv * H + head.  The
// constants are built on the host; total < 2^31 is checked there.
struct SlabGrid {
  FastDivmod per_lj;  // 2 * H * wps: sub-slabs per (layer, block)
  FastDivmod blocks;  // n_blocks
  FastDivmod heads;   // H
  uint32_t wps_log2;  // log2(block_size / 16)
  uint32_t total;     // sub-slabs in the call
  uint32_t units;     // ceil(total / 8): units of the persistent 8-warp CTAs
};

struct EncodeParams {
  SlabGrid grid;
  const void* k;
  const void* v;
  int64_t slot_stride;   // elements
  int64_t layer_stride;  // elements
  int32_t n_layers, H, B, num_slots, n_blocks, group, group_log2;
  const int32_t* src_slots;
  const int32_t* n_valid;  // may be null
  uint8_t* codes;
  void* scales;
  int32_t* err;
  // CRC-32 of every FP8 slab (its B x d codes, then its 4-byte scale), fused
  // into the encode when crc != null; the constants are built on the host
  // (see encode.cu, "Fused CRC").
  uint32_t* crc;
  uint32_t crc_sub[8];      // x^(8 * bytes from sub-slab k's end to the slab's codes' end)
  uint32_t crc_init;        // the initial register's term and the final xor
  // images of the single-bit inputs of the fused CRC's linear maps
  uint32_t crc_img_pos[8][64];    // pass i's 8 code bytes -> the lane's register at its last piece
  uint32_t crc_img_level[5][32];  // a register -> 8 * 2^j bytes later
  uint32_t crc_img_tail[32];      // a register -> 4 bytes later
  uint32_t crc_img_scale[32];     // the scale's 4 bytes -> the register after them
};

struct FetchParams {
  SlabGrid grid;
  const void* codes;
  const void* scales;
  const float* table;
  const int32_t* delta_idx;
  const int32_t* dst_slots;
  const int32_t* n_valid;  // may be null
  void* k;
  void* v;
  int64_t slot_stride, layer_stride;
  int32_t n_layers, H, B, num_slots, n_blocks, n_distinct, group, group_log2;
  int32_t* err;
};

struct TableParams {
  const int32_t* delta_m;
  const double* inv_freq;  // may be null: use theta[]
  float* table;
  int32_t n_distinct, half;
  double theta[128];
};

// CRC-32 of units a[u*a_stride ..+a_bytes) ++ b[u*b_stride ..+b_bytes), one
// warp per unit (crc32.cu): the unit's rows of 32 16-byte words, lane l
// taking word l of each row, kCrcGroup rows at a time, by persistent CTAs,
// kCrcCtasPerSm per SM; each lane moves its register of the 16-byte-word
// segment past the second segment (seg2_shift, img_seg2) and adds its
// register of the second, a butterfly over the lanes joins them, and
// init_term adds the initial register's contribution and the final xor.  Constants are built on the host.  Measured on GB300 over
// the Qwen3-8B-shaped FP8 wire (73,728 units of 32 KiB): groups of 4 rows at
// 8 CTAs/SM 3.43 TB/s (3.68 with the multiply-high field extraction and the
// scales read as words, 3.92 with one lane butterfly per unit and a grid of
// twice the nominal CTAs); at 4 CTAs/SM 3.17; groups of 8 rows 2.2-2.4.
#ifndef HC_CRC_GROUP
#define HC_CRC_GROUP 4
#endif
#ifndef HC_CRC_CTAS_PER_SM
#define HC_CRC_CTAS_PER_SM 8
#endif
constexpr int kCrcGroup = HC_CRC_GROUP;
constexpr int kCrcCtasPerSm = HC_CRC_CTAS_PER_SM;
// Units too few to fill the GPU one warp each are cut into chunks of at least
// this many groups (64 groups of 2 KiB: 128 KiB).
constexpr int kCrcMinChunkGroups = 64;
// The encoder's fused slab CRC with 16-token blocks: persistent CTAs, 2 per
// SM with the per-warp double buffer (128 registers), or 3-4 per SM with a
// single buffer (64 registers).  Measured on the Qwen3-8B-shaped encode
// (with the lane butterfly): 1.66 ms (2), 1.67 ms (3), 1.63 ms (4); the
// plain encode takes 1.08 ms.
#ifndef HC_FUSED_CRC_CTAS_PER_SM
#define HC_FUSED_CRC_CTAS_PER_SM 4
#endif
#ifndef HC_FUSED_CRC_WARPS
#define HC_FUSED_CRC_WARPS 8
#endif
constexpr int kFusedCrcCtasPerSm = HC_FUSED_CRC_CTAS_PER_SM;
constexpr int kFusedCrcWarps = HC_FUSED_CRC_WARPS;  // warps per persistent CTA (16 at most)

struct CrcParams {
  const uint8_t* a;
  const uint8_t* b;
  int64_t a_bytes, a_stride, b_bytes, b_stride;
  uint32_t n_units;
  uint32_t* crc;
  uint32_t seg2_shift;  // x^(8 * bytes of the second segment)
  int32_t b_words;      // the second segment is b alone, whole 16-byte words, 16-byte aligned
  uint32_t init_term;   // the initial register's term and the final xor
  // split launch (few, large units): chunks per unit, groups per chunk, and
  // x^(8 * bytes of 2^i groups)
  int64_t chunks, chunk_groups;
  uint32_t group_pow2[48];
  // images of the single-bit inputs of the kernel's linear maps (see crc32.cu)
  uint32_t img_word[kCrcGroup][128];
  uint32_t img_group[32];
  uint32_t img_level[5][32];
  uint32_t img_seg2[32];  // a register bit j times x^(8 * bytes of the second segment)
};

// Drift-ranked token selection over n_seq sequences of n_tokens rows of
// `hidden` elements (strides in elements).
struct SelectParams {
  const void* cached;
  const void* fresh;
  int64_t token_stride, seq_stride;
  int32_t n_seq, n_tokens, hidden, k;
  float* drift;       // [n_seq][n_tokens]
  int32_t* selected;  // [n_seq][k]
};

// Launchers: return the launch's cudaError_t.  `dtype`/`out_dtype` are hc_dtype.
cudaError_t launch_encode_fp8(int dtype, int d, const EncodeParams& p, cudaStream_t s);
// The FP8 encode with the fused slab CRC (16-bit sources; p.crc != null and
// the constants filled by make_slab_crc_constants).
cudaError_t launch_encode_fp8_crc(int dtype, int d, const EncodeParams& p, cudaStream_t s);
void make_slab_crc_constants(int d, int block_size, EncodeParams* p);
cudaError_t launch_encode_fp8_rows(int dtype, int d, bool scale_f16, const EncodeParams& p,
                                   cudaStream_t s);
cudaError_t launch_fetch_fp8_rows(int out_dtype, int d, bool half_split, bool scale_f16,
                                  const FetchParams& p, cudaStream_t s);
cudaError_t launch_crc32(const CrcParams& p, cudaStream_t s);
cudaError_t launch_drift_select(int dtype, const SelectParams& p, cudaStream_t s);
cudaError_t launch_encode_int4(int dtype, int d, bool scale_f16, const EncodeParams& p,
                               cudaStream_t s);
cudaError_t launch_fetch_fp8(int out_dtype, int d, bool half_split, const FetchParams& p,
                             cudaStream_t s);
cudaError_t launch_fetch_int4(int out_dtype, int d, bool half_split, bool scale_f16,
                              const FetchParams& p, cudaStream_t s);
cudaError_t launch_fetch_raw(int out_dtype, int d, bool half_split, const FetchParams& p,
                             cudaStream_t s);
cudaError_t launch_delta_table(const TableParams& p, cudaStream_t s);

// SlabGrid for a call; false if the call has 2^31 or more sub-slabs.
inline bool make_slab_grid(int64_t n_layers, int64_t n_blocks, int64_t H, int64_t B,
                           SlabGrid* g) {
  const int64_t wps = B / kRowsPerWarp;
  const int64_t total = n_layers * n_blocks * 2 * H * wps;
  if (n_blocks < 1 || total >= (int64_t{1} << 31)) return false;
  g->per_lj = FastDivmod(static_cast<uint32_t>(2 * H * wps));
  g->blocks = FastDivmod(static_cast<uint32_t>(n_blocks));
  g->heads = FastDivmod(static_cast<uint32_t>(H));
  g->wps_log2 = 0;
  while ((int64_t{1} << g->wps_log2) < wps) ++g->wps_log2;
  g->total = static_cast<uint32_t>(total);
  g->units = static_cast<uint32_t>((total + kWarps - 1) / kWarps);
  return true;
}

// Streaming multiprocessors of the current device (152 on GB300 if the query fails).
inline int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
    return n;
  return 152;
}


// ---------------------------------------------------------------- device side
#ifdef __CUDACC__

// Position of one warp's sub-slab, from the flat index (see SlabGrid).
struct Where {
  int64_t slab;  // wire slab index
  uint32_t l, j, kv, h, sub;
  bool active;   // index < total
};

__device__ __forceinline__ Where locate(const SlabGrid& g, uint32_t gw) {
  Where w;
  w.active = gw < g.total;
  const uint32_t n = w.active ? gw : 0u;
  uint32_t lj, u, slab_in_lj;
  g.per_lj.divmod(n, lj, u);
  g.blocks.divmod(lj, w.l, w.j);
  slab_in_lj = u >> g.wps_log2;
  w.sub = u - (slab_in_lj << g.wps_log2);
  g.heads.divmod(slab_in_lj, w.kv, w.h);
  w.slab = static_cast<int64_t>(lj) * (2 * g.heads.d) + slab_in_lj;
  return w;
}

// 8 consecutive elements of a source/destination dtype, kept as raw 16-byte words.
template <typename T>
struct Raw8 {
  static constexpr int kWords = sizeof(T) == 4 ? 2 : 1;
  uint4 w[kWords];
};

template <typename T>
__device__ __forceinline__ Raw8<T> load8_stream(const T* p) {
  Raw8<T> r;
#pragma unroll
  for (int i = 0; i < Raw8<T>::kWords; ++i) r.w[i] = __ldcs(reinterpret_cast<const uint4*>(p) + i);
  return r;
}

template <typename T>
__device__ __forceinline__ Raw8<T> raw8_zero() {
  Raw8<T> r;
#pragma unroll
  for (int i = 0; i < Raw8<T>::kWords; ++i) r.w[i] = make_uint4(0, 0, 0, 0);
  return r;
}

__device__ __forceinline__ float2 u32_to_float2(uint32_t u, const __half*) {
  __half2 h;
  memcpy(&h, &u, 4);
  return __half22float2(h);
}
__device__ __forceinline__ float2 u32_to_float2(uint32_t u, const __nv_bfloat16*) {
  __nv_bfloat162 h;
  memcpy(&h, &u, 4);
  return __bfloat1622float2(h);
}

template <typename T>
__device__ __forceinline__ void raw8_to_float(const Raw8<T>& r, float (&x)[8]) {
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      x[4 * i + 0] = __uint_as_float(r.w[i].x);
      x[4 * i + 1] = __uint_as_float(r.w[i].y);
      x[4 * i + 2] = __uint_as_float(r.w[i].z);
      x[4 * i + 3] = __uint_as_float(r.w[i].w);
    }
  } else {
    const uint32_t u[4] = {r.w[0].x, r.w[0].y, r.w[0].z, r.w[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = u32_to_float2(u[i], static_cast<const T*>(nullptr));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
}

// Running elementwise max of |x| over raw 16-byte words, kept packed:
// __half2 / __nv_bfloat162 lanes for 16-bit types, one float for fp32.
template <typename T>
struct AbsMax;
template <>
struct AbsMax<__half> {
  __half2 m = __float2half2_rn(0.f);
  __device__ __forceinline__ void add(const Raw8<__half>& r) {
    const uint4 w = r.w[0];
    __half2 a, b, c, d;
    memcpy(&a, &w.x, 4);
    memcpy(&b, &w.y, 4);
    memcpy(&c, &w.z, 4);
    memcpy(&d, &w.w, 4);
    m = __hmax2(m, __hmax2(__hmax2(__habs2(a), __habs2(b)), __hmax2(__habs2(c), __habs2(d))));
  }
  __device__ __forceinline__ float value() const {
    const float2 f = __half22float2(m);
    return fmaxf(f.x, f.y);
  }
};
template <>
struct AbsMax<__nv_bfloat16> {
  __nv_bfloat162 m = __float2bfloat162_rn(0.f);
  __device__ __forceinline__ void add(const Raw8<__nv_bfloat16>& r) {
    const uint4 w = r.w[0];
    __nv_bfloat162 a, b, c, d;
    memcpy(&a, &w.x, 4);
    memcpy(&b, &w.y, 4);
    memcpy(&c, &w.z, 4);
    memcpy(&d, &w.w, 4);
    m = __hmax2(m, __hmax2(__hmax2(__habs2(a), __habs2(b)), __hmax2(__habs2(c), __habs2(d))));
  }
  __device__ __forceinline__ float value() const {
    const float2 f = __bfloat1622float2(m);
    return fmaxf(f.x, f.y);
  }
};
template <>
struct AbsMax<float> {
  float m = 0.f;
  __device__ __forceinline__ void add(const Raw8<float>& r) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      m = fmaxf(m, fmaxf(fmaxf(fabsf(__uint_as_float(r.w[i].x)), fabsf(__uint_as_float(r.w[i].y))),
                         fmaxf(fabsf(__uint_as_float(r.w[i].z)), fabsf(__uint_as_float(r.w[i].w)))));
    }
  }
  __device__ __forceinline__ float value() const { return m; }
};

// 8 elements as 4 float2 (exact widening).
template <typename T>
__device__ __forceinline__ void raw8_to_float2(const Raw8<T>& r, float2 (&x)[4]) {
  float f[8];
  raw8_to_float(r, f);
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = make_float2(f[2 * i], f[2 * i + 1]);
}


__device__ __forceinline__ void flag_error(int32_t* err, int bits) {
  if (bits) atomicOr(err, bits);
}

#endif  // __CUDACC__

}  // namespace hc
