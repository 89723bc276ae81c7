/* A plain C client of libhc.so (test program): reads a case from a binary
 * file, runs encode (FP8), the delta-m table and the fetch through the C ABI
 * on cudaMalloc'd buffers, and writes codes, scales, the fetched K/V and the
 * error flag to an output file.
 *
 * Input file (little-endian): int32 L, H, d, B, S_src, S_dst, nb, n_distinct;
 * float64 rope_base; fp16 src_k[L][S_src][B][H][d], src_v[...]; int32
 * src_slots[nb], dst_slots[nb], n_valid[nb], delta_idx[nb];
 * int32 delta_m[n_distinct]; float32 dst_init[L][S_dst][B][H][d].
 * Output: u8 codes[L][nb][2][H][B][d]; f32 scales[L][nb][2][H];
 * f32 out_k[L][S_dst][B][H][d], out_v[...]; int32 err; u32 crc[L][nb] (the
 * CRC-32 of each (layer, block)'s codes followed by its scales); int32
 * hc_selection_size(1408).
 * Usage: hc_c_client <in> <out>; exit status 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "hc.h"

static void* read_n(FILE* f, size_t bytes) {
  void* p = malloc(bytes ? bytes : 1);
  if (!p || fread(p, 1, bytes, f) != bytes) {
    fprintf(stderr, "short read\n");
    exit(2);
  }
  return p;
}

static void* to_device(const void* h, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes ? bytes : 16) != cudaSuccess) exit(3);
  if (bytes && cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice) != cudaSuccess) exit(3);
  return d;
}

static void check(const char* what, int st) {
  if (st != HC_OK) {
    fprintf(stderr, "%s: %s %s\n", what, hc_status_string(st), hc_last_cuda_error());
    exit(4);
  }
}

int main(int argc, char** argv) {
  if (argc != 3) return 1;
  FILE* f = fopen(argv[1], "rb");
  if (!f) return 1;
  int32_t hdr[8];
  double rope_base;
  if (fread(hdr, 4, 8, f) != 8 || fread(&rope_base, 8, 1, f) != 1) return 2;
  const int32_t L = hdr[0], H = hdr[1], d = hdr[2], B = hdr[3], S_src = hdr[4], S_dst = hdr[5],
                nb = hdr[6], nd = hdr[7];
  const size_t src_elems = (size_t)L * S_src * B * H * d, dst_elems = (size_t)L * S_dst * B * H * d;
  void* h_k = read_n(f, src_elems * 2);
  void* h_v = read_n(f, src_elems * 2);
  void* h_src = read_n(f, (size_t)nb * 4);
  void* h_dst = read_n(f, (size_t)nb * 4);
  void* h_nv = read_n(f, (size_t)nb * 4);
  void* h_di = read_n(f, (size_t)nb * 4);
  void* h_dm = read_n(f, (size_t)nd * 4);
  void* h_init = read_n(f, dst_elems * 4);
  fclose(f);

  const size_t n_codes = (size_t)L * nb * 2 * H * B * d, n_scales = (size_t)L * nb * 2 * H;
  void *d_k = to_device(h_k, src_elems * 2), *d_v = to_device(h_v, src_elems * 2);
  void *d_src = to_device(h_src, (size_t)nb * 4), *d_dst = to_device(h_dst, (size_t)nb * 4);
  void *d_nv = to_device(h_nv, (size_t)nb * 4), *d_di = to_device(h_di, (size_t)nb * 4);
  void* d_dm = to_device(h_dm, (size_t)nd * 4);
  void *d_ok = to_device(h_init, dst_elems * 4), *d_ov = to_device(h_init, dst_elems * 4);
  void *d_codes = NULL, *d_scales = NULL, *d_table = NULL, *d_err = NULL, *d_crc = NULL;
  if (cudaMalloc(&d_codes, n_codes) || cudaMalloc(&d_scales, n_scales * 4) ||
      cudaMalloc(&d_table, (size_t)nd * d * 4) || cudaMalloc(&d_err, 4) || cudaMemset(d_err, 0, 4) ||
      cudaMalloc(&d_crc, (size_t)L * nb * 4))
    return 3;

  hc_paged_desc src = {L, H, d, B, S_src, HC_F16, (int64_t)B * H * d, (int64_t)S_src * B * H * d};
  hc_paged_desc dst = {L, H, d, B, S_dst, HC_F32, (int64_t)B * H * d, (int64_t)S_dst * B * H * d};
  check("hc_encode_fp8", hc_encode_fp8(d_k, d_v, &src, (const int32_t*)d_src, (const int32_t*)d_nv,
                                       nb, (uint8_t*)d_codes, (float*)d_scales, (int32_t*)d_err, NULL));
  check("hc_build_delta_sincos", hc_build_delta_sincos((const int32_t*)d_dm, nd, d, rope_base, NULL,
                                                       (float*)d_table, NULL));
  check("hc_fetch_rotate_scatter",
        hc_fetch_rotate_scatter(HC_WIRE_FP8, d_codes, d_scales, 32, HC_F16, (const float*)d_table,
                                (const int32_t*)d_di, nd, HC_PAIR_HALF_SPLIT, (const int32_t*)d_dst,
                                (const int32_t*)d_nv, nb, d_ok, d_ov, &dst, (int32_t*)d_err, NULL));
  {
    const int64_t unit_codes = (int64_t)2 * H * B * d, unit_scales = (int64_t)2 * H * 4;
    check("hc_crc32", hc_crc32(d_codes, unit_codes, unit_codes, d_scales, unit_scales, unit_scales,
                               L * nb, (uint32_t*)d_crc, NULL));
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return 5;

  uint8_t* codes = (uint8_t*)malloc(n_codes);
  float* scales = (float*)malloc(n_scales * 4);
  float* ok = (float*)malloc(dst_elems * 4);
  float* ov = (float*)malloc(dst_elems * 4);
  int32_t err = -1;
  uint32_t* crc = (uint32_t*)malloc((size_t)L * nb * 4);
  if (cudaMemcpy(crc, d_crc, (size_t)L * nb * 4, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(codes, d_codes, n_codes, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(scales, d_scales, n_scales * 4, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(ok, d_ok, dst_elems * 4, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(ov, d_ov, dst_elems * 4, cudaMemcpyDeviceToHost) ||
      cudaMemcpy(&err, d_err, 4, cudaMemcpyDeviceToHost))
    return 5;
  FILE* o = fopen(argv[2], "wb");
  if (!o) return 6;
  fwrite(codes, 1, n_codes, o);
  fwrite(scales, 4, n_scales, o);
  fwrite(ok, 4, dst_elems, o);
  fwrite(ov, 4, dst_elems, o);
  fwrite(&err, 4, 1, o);
  fwrite(crc, 4, (size_t)L * nb, o);
  const int32_t k_default = hc_selection_size(1408);
  fwrite(&k_default, 4, 1, o);
  fclose(o);
  printf("hc_c_client: ok (library API version %d)\n", hc_version());
  return 0;
}
