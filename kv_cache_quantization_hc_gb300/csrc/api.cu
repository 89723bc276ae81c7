// C ABI entry points: host-side validation, then one kernel launch on the
// caller's stream.  No allocation, no synchronization, no global state except
// the per-thread text of the last CUDA error.
#include <cmath>
#include <cstdio>
#include <cstring>

#include "hc_internal.cuh"

namespace {

thread_local char g_last_cuda_error[256] = "";

int record(cudaError_t e) {
  if (e == cudaSuccess) return HC_OK;
  std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return HC_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_size(int dtype) {
  switch (dtype) {
    case HC_F32: return 4;
    case HC_F16: return 2;
    case HC_BF16: return 2;
  }
  return 0;
}

// Validates a paged descriptor and the two buffer bases.
int check_paged(const hc_paged_desc* d, const void* k, const void* v) {
  if (!d || !k || !v) return HC_ERR_INVALID_ARG;
  const int es = elem_size(d->dtype);
  if (es == 0) return HC_ERR_INVALID_ARG;
  if (d->n_layers < 1 || d->n_kv_heads < 1 || d->num_slots < 1 || d->d_head < 1 ||
      d->block_size < 1)
    return HC_ERR_INVALID_ARG;
  if (d->d_head != 64 && d->d_head != 128) return HC_ERR_UNSUPPORTED;
  if (d->block_size != 16 && d->block_size != 32 && d->block_size != 64 && d->block_size != 128)
    return HC_ERR_UNSUPPORTED;
  const int64_t slot_elems = static_cast<int64_t>(d->block_size) * d->n_kv_heads * d->d_head;
  if (d->slot_stride < slot_elems) return HC_ERR_INVALID_ARG;
  if (d->layer_stride < 0 || (d->n_layers > 1 && d->layer_stride == 0)) return HC_ERR_INVALID_ARG;
  if ((d->slot_stride * es) % 16 || (d->layer_stride * es) % 16) return HC_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16)) return HC_ERR_INVALID_ARG;
  return HC_OK;
}

// The kernels index sub-slabs with 32-bit arithmetic: fewer than 2^31 per call.
bool grid_fits(const hc_paged_desc* d, int32_t n_blocks) {
  hc::SlabGrid g;
  return n_blocks == 0 || hc::make_slab_grid(d->n_layers, n_blocks, d->n_kv_heads, d->block_size, &g);
}

hc::EncodeParams encode_params(const void* k, const void* v, const hc_paged_desc* d,
                               const int32_t* src, const int32_t* nv, int32_t nb, uint8_t* codes,
                               void* scales, int32_t* err, int32_t group) {
  hc::EncodeParams p;
  hc::make_slab_grid(d->n_layers, nb, d->n_kv_heads, d->block_size, &p.grid);
  p.k = k;
  p.v = v;
  p.slot_stride = d->slot_stride;
  p.layer_stride = d->layer_stride;
  p.n_layers = d->n_layers;
  p.H = d->n_kv_heads;
  p.B = d->block_size;
  p.num_slots = d->num_slots;
  p.n_blocks = nb;
  p.group = group;
  p.group_log2 = group == 128 ? 7 : group == 64 ? 6 : 5;
  p.src_slots = src;
  p.n_valid = nv;
  p.codes = codes;
  p.scales = scales;
  p.err = err;
  p.crc = nullptr;
  return p;
}

}  // namespace

extern "C" {

int hc_encode_fp8(const void* paged_k, const void* paged_v, const hc_paged_desc* desc,
                  const int32_t* src_slots, const int32_t* n_valid, int32_t n_blocks,
                  uint8_t* codes, float* scales, int32_t* err_flag, void* stream) {
  int st = check_paged(desc, paged_k, paged_v);
  if (st != HC_OK) return st;
  if (n_blocks < 0) return HC_ERR_INVALID_ARG;
  if (!src_slots || !codes || !scales || !err_flag) return HC_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(scales, 4) || !aligned(err_flag, 4) ||
      !aligned(src_slots, 4) || (n_valid && !aligned(n_valid, 4)))
    return HC_ERR_INVALID_ARG;
  if (!grid_fits(desc, n_blocks)) return HC_ERR_INVALID_ARG;
  if (n_blocks == 0) return HC_OK;
  const hc::EncodeParams p = encode_params(paged_k, paged_v, desc, src_slots, n_valid, n_blocks,
                                           codes, scales, err_flag, 0);
  return record(hc::launch_encode_fp8(desc->dtype, desc->d_head, p,
                                      static_cast<cudaStream_t>(stream)));
}

int hc_encode_fp8_crc(const void* paged_k, const void* paged_v, const hc_paged_desc* desc,
                      const int32_t* src_slots, const int32_t* n_valid, int32_t n_blocks,
                      uint8_t* codes, float* scales, uint32_t* crc, int32_t* err_flag,
                      void* stream) {
  if (!crc || !aligned(crc, 4)) return HC_ERR_INVALID_ARG;
  int st = check_paged(desc, paged_k, paged_v);
  if (st != HC_OK) return st;
  if (n_blocks < 0) return HC_ERR_INVALID_ARG;
  if (!src_slots || !codes || !scales || !err_flag) return HC_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(scales, 4) || !aligned(err_flag, 4) ||
      !aligned(src_slots, 4) || (n_valid && !aligned(n_valid, 4)))
    return HC_ERR_INVALID_ARG;
  if (!grid_fits(desc, n_blocks)) return HC_ERR_INVALID_ARG;
  if (n_blocks == 0) return HC_OK;
  hc::EncodeParams p = encode_params(paged_k, paged_v, desc, src_slots, n_valid, n_blocks, codes,
                                     scales, err_flag, 0);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (desc->dtype == HC_F32) {
    // fp32 sources: the encode, then the CRC kernel over the same slab units
    st = record(hc::launch_encode_fp8(desc->dtype, desc->d_head, p, s));
    if (st != HC_OK) return st;
    const int64_t slab = int64_t{desc->block_size} * desc->d_head;
    return hc_crc32(codes, slab, slab, scales, 4, 4,
                    static_cast<int32_t>(int64_t{desc->n_layers} * n_blocks * 2 * desc->n_kv_heads),
                    crc, stream);
  }
  p.crc = crc;
  hc::make_slab_crc_constants(desc->d_head, desc->block_size, &p);
  return record(hc::launch_encode_fp8_crc(desc->dtype, desc->d_head, p, s));
}

int hc_encode_int4(const void* paged_k, const void* paged_v, const hc_paged_desc* desc,
                   const int32_t* src_slots, const int32_t* n_valid, int32_t n_blocks,
                   int32_t group, int32_t scale_dtype, uint8_t* codes, void* scales,
                   int32_t* err_flag, void* stream) {
  int st = check_paged(desc, paged_k, paged_v);
  if (st != HC_OK) return st;
  if (n_blocks < 0) return HC_ERR_INVALID_ARG;
  if (!src_slots || !codes || !scales || !err_flag) return HC_ERR_INVALID_ARG;
  if (scale_dtype != HC_F16 && scale_dtype != HC_F32) return HC_ERR_INVALID_ARG;
  if (group != 32 && group != 64 && group != 128) return HC_ERR_UNSUPPORTED;
  if (group > desc->d_head) return HC_ERR_UNSUPPORTED;
  if (!aligned(codes, 16) || !aligned(scales, scale_dtype == HC_F16 ? 2 : 4) ||
      !aligned(err_flag, 4) || !aligned(src_slots, 4) || (n_valid && !aligned(n_valid, 4)))
    return HC_ERR_INVALID_ARG;
  if (!grid_fits(desc, n_blocks)) return HC_ERR_INVALID_ARG;
  if (n_blocks == 0) return HC_OK;
  const hc::EncodeParams p = encode_params(paged_k, paged_v, desc, src_slots, n_valid, n_blocks,
                                           codes, scales, err_flag, group);
  return record(hc::launch_encode_int4(desc->dtype, desc->d_head, scale_dtype == HC_F16, p,
                                       static_cast<cudaStream_t>(stream)));
}

int hc_encode_fp8_rows(const void* paged_k, const void* paged_v, const hc_paged_desc* desc,
                       const int32_t* src_slots, const int32_t* n_valid, int32_t n_blocks,
                       int32_t scale_dtype, uint8_t* codes, void* scales, int32_t* err_flag,
                       void* stream) {
  int st = check_paged(desc, paged_k, paged_v);
  if (st != HC_OK) return st;
  if (n_blocks < 0) return HC_ERR_INVALID_ARG;
  if (!src_slots || !codes || !scales || !err_flag) return HC_ERR_INVALID_ARG;
  if (scale_dtype != HC_F16 && scale_dtype != HC_F32) return HC_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(scales, scale_dtype == HC_F16 ? 2 : 4) ||
      !aligned(err_flag, 4) || !aligned(src_slots, 4) || (n_valid && !aligned(n_valid, 4)))
    return HC_ERR_INVALID_ARG;
  if (!grid_fits(desc, n_blocks)) return HC_ERR_INVALID_ARG;
  if (n_blocks == 0) return HC_OK;
  const hc::EncodeParams p = encode_params(paged_k, paged_v, desc, src_slots, n_valid, n_blocks,
                                           codes, scales, err_flag, 0);
  return record(hc::launch_encode_fp8_rows(desc->dtype, desc->d_head, scale_dtype == HC_F16, p,
                                           static_cast<cudaStream_t>(stream)));
}

int hc_build_delta_sincos(const int32_t* delta_m, int32_t n_distinct, int32_t d_head,
                          double rope_base, const double* inv_freq, float* table,
                          void* stream) {
  if (n_distinct < 0 || d_head < 2 || d_head > 256 || (d_head & 1)) return HC_ERR_INVALID_ARG;
  if (!delta_m || !table) return HC_ERR_INVALID_ARG;
  if (!inv_freq && !(rope_base > 0.0 && std::isfinite(rope_base))) return HC_ERR_INVALID_ARG;
  if (!aligned(table, 16) || !aligned(delta_m, 4) || (inv_freq && !aligned(inv_freq, 8)))
    return HC_ERR_INVALID_ARG;
  if (n_distinct == 0) return HC_OK;
  hc::TableParams p;
  std::memset(&p, 0, sizeof p);
  p.delta_m = delta_m;
  p.inv_freq = inv_freq;
  p.table = table;
  p.n_distinct = n_distinct;
  p.half = d_head / 2;
  if (!inv_freq) {
    // theta_i = base^(-2i/d), the same fp64 expression as the rope_cache
    // listing, evaluated by the C library's pow.
    for (int i = 0; i < p.half; ++i) p.theta[i] = std::pow(rope_base, -(2.0 * i) / d_head);
  }
  return record(hc::launch_delta_table(p, static_cast<cudaStream_t>(stream)));
}

int hc_fetch_rotate_scatter(int32_t wire, const void* codes, const void* scales, int32_t group,
                            int32_t scale_dtype, const float* table, const int32_t* delta_idx,
                            int32_t n_distinct, int32_t pairing, const int32_t* dst_slots,
                            const int32_t* n_valid, int32_t n_blocks, void* paged_k,
                            void* paged_v, const hc_paged_desc* desc, int32_t* err_flag,
                            void* stream) {
  int st = check_paged(desc, paged_k, paged_v);
  if (st != HC_OK) return st;
  if (n_blocks < 0) return HC_ERR_INVALID_ARG;
  if (wire != HC_WIRE_FP8 && wire != HC_WIRE_INT4 && wire != HC_WIRE_RAW &&
      wire != HC_WIRE_FP8_ROWS)
    return HC_ERR_INVALID_ARG;
  if (pairing != HC_PAIR_INTERLEAVED && pairing != HC_PAIR_HALF_SPLIT) return HC_ERR_INVALID_ARG;
  if (!codes || !table || !delta_idx || !dst_slots || !err_flag) return HC_ERR_INVALID_ARG;
  if (wire != HC_WIRE_RAW && !scales) return HC_ERR_INVALID_ARG;
  if (n_blocks > 0 && n_distinct < 1) return HC_ERR_INVALID_ARG;
  if (wire == HC_WIRE_INT4) {
    if (scale_dtype != HC_F16 && scale_dtype != HC_F32) return HC_ERR_INVALID_ARG;
    if (group != 32 && group != 64 && group != 128) return HC_ERR_UNSUPPORTED;
    if (group > desc->d_head) return HC_ERR_UNSUPPORTED;
    if (!aligned(scales, scale_dtype == HC_F16 ? 2 : 4)) return HC_ERR_INVALID_ARG;
  }
  if (wire == HC_WIRE_FP8 && !aligned(scales, 4)) return HC_ERR_INVALID_ARG;
  if (wire == HC_WIRE_FP8_ROWS) {
    if (scale_dtype != HC_F16 && scale_dtype != HC_F32) return HC_ERR_INVALID_ARG;
    if (!aligned(scales, scale_dtype == HC_F16 ? 2 : 4)) return HC_ERR_INVALID_ARG;
  }
  if (!aligned(codes, 16) || !aligned(table, 16) || !aligned(delta_idx, 4) ||
      !aligned(dst_slots, 4) || !aligned(err_flag, 4) || (n_valid && !aligned(n_valid, 4)))
    return HC_ERR_INVALID_ARG;
  if (!grid_fits(desc, n_blocks)) return HC_ERR_INVALID_ARG;
  if (n_blocks == 0) return HC_OK;

  hc::FetchParams p;
  hc::make_slab_grid(desc->n_layers, n_blocks, desc->n_kv_heads, desc->block_size, &p.grid);
  p.codes = codes;
  p.scales = scales;
  p.table = table;
  p.delta_idx = delta_idx;
  p.dst_slots = dst_slots;
  p.n_valid = n_valid;
  p.k = paged_k;
  p.v = paged_v;
  p.slot_stride = desc->slot_stride;
  p.layer_stride = desc->layer_stride;
  p.n_layers = desc->n_layers;
  p.H = desc->n_kv_heads;
  p.B = desc->block_size;
  p.num_slots = desc->num_slots;
  p.n_blocks = n_blocks;
  p.n_distinct = n_distinct;
  p.group = group;
  p.group_log2 = group == 128 ? 7 : group == 64 ? 6 : 5;
  p.err = err_flag;
  const bool half = pairing == HC_PAIR_HALF_SPLIT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (wire) {
    case HC_WIRE_FP8: return record(hc::launch_fetch_fp8(desc->dtype, desc->d_head, half, p, s));
    case HC_WIRE_INT4:
      return record(
          hc::launch_fetch_int4(desc->dtype, desc->d_head, half, scale_dtype == HC_F16, p, s));
    case HC_WIRE_FP8_ROWS:
      return record(hc::launch_fetch_fp8_rows(desc->dtype, desc->d_head, half,
                                              scale_dtype == HC_F16, p, s));
    default: return record(hc::launch_fetch_raw(desc->dtype, desc->d_head, half, p, s));
  }
}

int hc_crc32(const void* a, int64_t a_bytes, int64_t a_stride, const void* b, int64_t b_bytes,
             int64_t b_stride, int32_t n_units, uint32_t* crc, void* stream) {
  if (n_units < 0 || a_bytes < 0 || b_bytes < 0 || a_stride < 0 || b_stride < 0)
    return HC_ERR_INVALID_ARG;
  if (!crc || (a_bytes > 0 && !a) || (b_bytes > 0 && !b)) return HC_ERR_INVALID_ARG;
  if ((a && !aligned(a, 16)) || a_stride % 16 || !aligned(crc, 4)) return HC_ERR_INVALID_ARG;
  if (n_units > 1 && (a_stride < a_bytes || (b_bytes > 0 && b_stride < b_bytes)))
    return HC_ERR_INVALID_ARG;
  if (n_units == 0) return HC_OK;
  hc::CrcParams p;
  std::memset(&p, 0, sizeof p);
  p.a = static_cast<const uint8_t*>(a);
  p.b = static_cast<const uint8_t*>(b);
  p.a_bytes = a_bytes;
  p.a_stride = a_stride;
  p.b_bytes = b_bytes;
  p.b_stride = b_stride;
  p.n_units = static_cast<uint32_t>(n_units);
  p.crc = crc;
  return record(hc::launch_crc32(p, static_cast<cudaStream_t>(stream)));
}

int32_t hc_selection_size(int32_t n_tokens) {
  // ceil(15% of n_tokens) in integers: 15/100 = 3/20; n_tokens < 2^31 keeps
  // 3 * n_tokens + 19 inside int64.
  if (n_tokens < 1) return 0;
  return static_cast<int32_t>((int64_t{3} * n_tokens + 19) / 20);
}

int hc_drift_select(const void* h_cached, const void* h_fresh, int32_t dtype, int32_t n_seq,
                    int32_t n_tokens, int32_t hidden, int64_t token_stride, int64_t seq_stride,
                    int32_t k, float* drift, int32_t* selected, void* stream) {
  const int es = elem_size(dtype);
  if (es == 0 || n_seq < 0 || n_tokens < 1 || hidden < 8 || hidden % 8) return HC_ERR_INVALID_ARG;
  if (k <= 0) k = hc_selection_size(n_tokens);
  if (k > n_tokens) return HC_ERR_INVALID_ARG;
  if (!h_cached || !h_fresh || !drift || !selected) return HC_ERR_INVALID_ARG;
  if (token_stride < hidden || (n_seq > 1 && seq_stride < int64_t{n_tokens} * token_stride))
    return HC_ERR_INVALID_ARG;
  if ((token_stride * es) % 16 || (seq_stride * es) % 16 || seq_stride < 0) return HC_ERR_INVALID_ARG;
  if (!aligned(h_cached, 16) || !aligned(h_fresh, 16) || !aligned(drift, 4) || !aligned(selected, 4))
    return HC_ERR_INVALID_ARG;
  if (int64_t{n_seq} * n_tokens >= (int64_t{1} << 31)) return HC_ERR_INVALID_ARG;
  if (n_seq == 0) return HC_OK;
  hc::SelectParams p;
  p.cached = h_cached;
  p.fresh = h_fresh;
  p.token_stride = token_stride;
  p.seq_stride = seq_stride;
  p.n_seq = n_seq;
  p.n_tokens = n_tokens;
  p.hidden = hidden;
  p.k = k;
  p.drift = drift;
  p.selected = selected;
  return record(hc::launch_drift_select(dtype, p, static_cast<cudaStream_t>(stream)));
}

const char* hc_status_string(int32_t status) {
  switch (status) {
    case HC_OK: return "HC_OK";
    case HC_ERR_INVALID_ARG: return "HC_ERR_INVALID_ARG";
    case HC_ERR_UNSUPPORTED: return "HC_ERR_UNSUPPORTED";
    case HC_ERR_CUDA: return "HC_ERR_CUDA";
  }
  return "HC_UNKNOWN_STATUS";
}

const char* hc_last_cuda_error(void) { return g_last_cuda_error; }

int32_t hc_version(void) { return HC_API_VERSION; }

}  // extern "C"
