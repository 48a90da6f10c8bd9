// Load-time weight repacking, its inverse, the test dequantiser, and the f16 /
// bf16 conversions.
//
// The pages' loaders hand each block to the GPU as it sits in the model file
// (an 18-, 20-, 22-, 34-, 144-, 176- or 210-byte record).  Those records are not
// 16-byte aligned, so the repack splits every tensor into a code region (16 B per
// Q4_0 / Q4_1 / Q5_0 block, 32 B per Q8_0 block, 128 / 160 / 192 B per Q4_K / Q5_K /
// Q6_K super-block, one byte per INT8 weight, two per F16 weight) and a scale region
// (the rest of each record: f16 d, d and m, d and qh, the 16-byte d/dmin/scales header,
// Q6_K's 16 scales and d; one f32 per INT8 row; nothing for F16), both row-major.  Nothing is re-encoded:
// the scales stay f16 (the Go "llm" package's "Design points" widen them to f32
// only because its shading language has no f16), so the packed tensor is the
// same number of bytes as the source plus at most 30 bytes of padding.
#include "qd_internal.cuh"

namespace qd {
namespace {

struct BlockGeom {
  int src_bytes;    // bytes of one source block
  int weights;      // weights per block
  int code_off;     // offset of the codes inside the source block
  int code_bytes;   // bytes of codes per block
  int scale_off;    // offset of the scale data inside the source block
  int scale_bytes;  // bytes of scale data per block
};

__host__ __device__ inline BlockGeom geom(int fmt) {
  switch (fmt) {
    case QD_Q4_0: return {18, 32, 2, 16, 0, 2};
    case QD_Q8_0: return {34, 32, 2, 32, 0, 2};
    case QD_Q4_1: return {20, 32, 4, 16, 0, 4};      // d, m | codes
    case QD_Q5_0: return {22, 32, 6, 16, 0, 6};      // d, qh | low nibbles
    case QD_Q5_K: return {176, 256, 16, 160, 0, 16};  // d, dmin, scales | qh, low nibbles
    case QD_Q6_K: return {210, 256, 0, 192, 192, 18};  // ql, qh | scales, d
    case QD_F16: return {32, 16, 0, 32, 0, 0};       // 16 weights as one "block"
    default: return {144, 256, 16, 128, 0, 16};       // QD_Q4_K
  }
}

// Destination row of source row i (see launch_repack_rows).
__host__ __device__ inline int64_t dst_row_of(int64_t i, int64_t row0, int64_t step, int pair_hd) {
  if (pair_hd > 0) {
    const int64_t h = i / pair_hd, l = i % pair_hd, half = pair_hd / 2;
    i = h * pair_hd + 2 * (l % half) + l / half;
  }
  return row0 + i * step;
}

// One thread per (source row, block): copy its codes and its scale bytes.
__global__ void k_repack_blocks(int fmt, const uint8_t* __restrict__ src, int64_t n_rows, int64_t nb,
                                uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int64_t dst_row0,
                                int64_t dst_step, int pair_hd) {
  const BlockGeom g = geom(fmt);
  const int64_t total = n_rows * nb;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = t / nb, b = t % nb;
    const int64_t r = dst_row_of(i, dst_row0, dst_step, pair_hd);
    const uint8_t* s = src + t * g.src_bytes;
    uint8_t* c = codes + (r * nb + b) * g.code_bytes;
    uint8_t* sc = scales + (r * nb + b) * g.scale_bytes;
    for (int k = 0; k < g.code_bytes; ++k) c[k] = s[g.code_off + k];
    for (int k = 0; k < g.scale_bytes; ++k) sc[k] = s[g.scale_off + k];
  }
}

__global__ void k_unpack_blocks(int fmt, const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                int64_t rows, int64_t nb, uint8_t* __restrict__ dst) {
  const BlockGeom g = geom(fmt);
  const int64_t total = rows * nb;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    uint8_t* d = dst + t * g.src_bytes;
    const uint8_t* c = codes + t * g.code_bytes;
    const uint8_t* sc = scales + t * g.scale_bytes;
    for (int k = 0; k < g.scale_bytes; ++k) d[g.scale_off + k] = sc[k];
    for (int k = 0; k < g.code_bytes; ++k) d[g.code_off + k] = c[k];
  }
}

// INT8 rows: codes copy 16 bytes per thread, scales one f32 per row.
__global__ void k_repack_i8(const uint8_t* __restrict__ src, int64_t n_rows, int64_t cols,
                            uint8_t* __restrict__ codes, float* __restrict__ scales, int64_t dst_row0,
                            int64_t dst_step, int pair_hd) {
  const int64_t chunks = cols / 16;
  const int64_t total = n_rows * chunks;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = t / chunks, c = t % chunks;
    const int64_t r = dst_row_of(i, dst_row0, dst_step, pair_hd);
    const uint8_t* s = src + i * cols + c * 16;
    uint8_t* d = codes + r * cols + c * 16;
    for (int k = 0; k < 16; ++k) d[k] = s[k];  // source rows are only byte-aligned in general
    if (c == 0) {
      float v;
      memcpy(&v, src + n_rows * cols + 4 * i, 4);
      scales[r] = v;
    }
  }
}

// INT4 rows: the source holds element 2i in the low nibble of byte i (two's complement);
// the packed codes hold each 32-element unit as Q4_0 orders it (element j in the low
// nibble of byte j, element j + 16 in its high nibble) in offset binary (q + 8), which the
// streaming GEMV's Q4_0 path reads.  One thread per (source row, unit).
__device__ __forceinline__ int src_i4_nibble(const uint8_t* unit, int e) { return (unit[e >> 1] >> (4 * (e & 1))) & 15; }

__global__ void k_repack_i4(const uint8_t* __restrict__ src, int64_t n_rows, int64_t cols, uint8_t* __restrict__ codes,
                            float* __restrict__ scales, int64_t dst_row0, int64_t dst_step, int pair_hd) {
  const int64_t units = cols / 32, total = n_rows * units;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = t / units, u = t % units;
    const int64_t r = dst_row_of(i, dst_row0, dst_step, pair_hd);
    const uint8_t* s = src + i * (cols / 2) + 16 * u;
    uint8_t* d = codes + r * (cols / 2) + 16 * u;
    for (int j = 0; j < 16; ++j)
      d[j] = (uint8_t)((src_i4_nibble(s, j) ^ 8) | ((src_i4_nibble(s, j + 16) ^ 8) << 4));
    if (u == 0) {
      float v;
      memcpy(&v, src + n_rows * (cols / 2) + 4 * i, 4);
      scales[r] = v;
    }
  }
}

__global__ void k_unpack_i4(const uint8_t* __restrict__ codes, const float* __restrict__ scales, int64_t rows,
                            int64_t cols, uint8_t* __restrict__ dst) {
  const int64_t units = cols / 32, total = rows * units;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const uint8_t* c = codes + 16 * t;  // unit u of row r = t / units, rows contiguous
    uint8_t* d = dst + 16 * t;
    for (int i = 0; i < 16; ++i) {  // source byte i: elements 2i, 2i + 1
      int nib[2];
      for (int h = 0; h < 2; ++h) {
        const int e = 2 * i + h;
        nib[h] = ((e < 16 ? c[e] : c[e - 16] >> 4) & 15) ^ 8;
      }
      d[i] = (uint8_t)(nib[0] | (nib[1] << 4));
    }
    if (t % units == 0) {
      const float v = scales[t / units];
      memcpy(dst + rows * (cols / 2) + 4 * (t / units), &v, 4);
    }
  }
}

__global__ void k_unpack_i8(const uint8_t* __restrict__ codes, const float* __restrict__ scales, int64_t rows,
                            int64_t cols, uint8_t* __restrict__ dst) {
  const int64_t total = rows * cols;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    dst[t] = codes[t];
    if (t % cols == 0) {
      const float v = scales[t / cols];
      memcpy(dst + total + 4 * (t / cols), &v, 4);
    }
  }
}

__global__ void k_dequant(int fmt, PackedView W, float* __restrict__ out) {
  const int64_t total = W.rows * W.cols;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x)
    out[t] = dequant_elem(fmt, W, t / W.cols, t % W.cols);
}

__global__ void k_f16_to_f32(const uint16_t* __restrict__ in, float* __restrict__ out, int64_t n) {
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x)
    out[t] = f16_bits_to_f32(in[t]);
}

// bf16 -> f32 is the zero-extension of the bit pattern (minillm-cpp README, "Loader").
__global__ void k_bf16_to_f32(const uint16_t* __restrict__ in, float* __restrict__ out, int64_t n) {
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x)
    out[t] = __uint_as_float((uint32_t)in[t] << 16);
}

inline int grid_for(int64_t n, int threads) {
  int64_t g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  return (int)(g > 65535 * 8 ? 65535 * 8 : g);
}

}  // namespace

qd_status launch_repack_rows(int fmt, const void* src, int64_t n_rows, int64_t cols, void* dst_base,
                             int64_t dst_rows, int64_t dst_row0, int64_t dst_row_step, cudaStream_t stream,
                             int pair_hd) {
  if (pair_hd > 0 && ((pair_hd & 1) || n_rows % pair_hd)) return QD_ERR_SHAPE;
  PackedView v = packed_view(fmt, dst_base, dst_rows, cols);
  uint8_t* codes = const_cast<uint8_t*>(v.codes);
  uint8_t* scales = const_cast<uint8_t*>(v.scales);
  if (fmt == QD_I4_ROW) {
    k_repack_i4<<<grid_for(n_rows * (cols / 32), 256), 256, 0, stream>>>(
        static_cast<const uint8_t*>(src), n_rows, cols, codes, reinterpret_cast<float*>(scales), dst_row0,
        dst_row_step, pair_hd);
  } else if (fmt == QD_I8_ROW) {  // codes row by row, then one f32 scale per row
    const int64_t rb = row_code_bytes(fmt, cols);
    const int64_t n = n_rows * (rb / 16);
    k_repack_i8<<<grid_for(n, 256), 256, 0, stream>>>(static_cast<const uint8_t*>(src), n_rows, rb, codes,
                                                       reinterpret_cast<float*>(scales), dst_row0, dst_row_step,
                                                       pair_hd);
  } else {
    const int64_t nb = cols / geom(fmt).weights;
    k_repack_blocks<<<grid_for(n_rows * nb, 256), 256, 0, stream>>>(fmt, static_cast<const uint8_t*>(src), n_rows,
                                                                    nb, codes, scales, dst_row0, dst_row_step,
                                                                    pair_hd);
  }
  return launch_status();
}

}  // namespace qd

using namespace qd;

extern "C" {

const char* qd_status_str(qd_status s) {
  switch (s) {
    case QD_OK: return "ok";
    case QD_ERR_INVALID_ARG: return "invalid argument";
    case QD_ERR_SHAPE: return "shape not allowed";
    case QD_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case QD_ERR_UNSUPPORTED: return "unsupported format or configuration";
    case QD_ERR_CUDA: return "CUDA error";
    case QD_ERR_NOMEM: return "buffer too small";
    case QD_ERR_DEVICE_FLAG: return "a kernel flagged an out-of-range token or position";
    default: return "unknown status";
  }
}

int qd_abi_version(void) { return 4; }

size_t qd_src_bytes(qd_fmt fmt, int64_t rows, int64_t cols) { return src_bytes(fmt, rows, cols); }
size_t qd_packed_bytes(qd_fmt fmt, int64_t rows, int64_t cols) { return packed_bytes(fmt, rows, cols); }

qd_status qd_repack(qd_fmt fmt, const void* src, int64_t rows, int64_t cols, void* dst, size_t dst_bytes,
                    qd_stream_t stream) {
  if (!fmt_ok(fmt)) return QD_ERR_UNSUPPORTED;
  if (!src || !dst) return QD_ERR_INVALID_ARG;
  if (!shape_ok(fmt, rows, cols)) return QD_ERR_SHAPE;
  if (!aligned16(dst)) return QD_ERR_ALIGN;
  if (dst_bytes < packed_bytes(fmt, rows, cols)) return QD_ERR_NOMEM;
  return launch_repack_rows(fmt, src, rows, cols, dst, rows, 0, 1, (cudaStream_t)stream);
}

qd_status qd_unpack(qd_fmt fmt, const void* packed, int64_t rows, int64_t cols, void* dst, size_t dst_bytes,
                    qd_stream_t stream) {
  if (!fmt_ok(fmt)) return QD_ERR_UNSUPPORTED;
  if (!packed || !dst) return QD_ERR_INVALID_ARG;
  if (!shape_ok(fmt, rows, cols)) return QD_ERR_SHAPE;
  if (!aligned16(packed)) return QD_ERR_ALIGN;
  if (dst_bytes < src_bytes(fmt, rows, cols)) return QD_ERR_NOMEM;
  PackedView v = packed_view(fmt, packed, rows, cols);
  cudaStream_t s = (cudaStream_t)stream;
  if (fmt == QD_I4_ROW) {
    k_unpack_i4<<<grid_for(rows * (cols / 32), 256), 256, 0, s>>>(v.codes, reinterpret_cast<const float*>(v.scales),
                                                                  rows, cols, static_cast<uint8_t*>(dst));
  } else if (fmt == QD_I8_ROW) {
    k_unpack_i8<<<grid_for(rows * cols, 256), 256, 0, s>>>(v.codes, reinterpret_cast<const float*>(v.scales), rows,
                                                            cols, static_cast<uint8_t*>(dst));
  } else {
    const int64_t nb = cols / geom(fmt).weights;
    k_unpack_blocks<<<grid_for(rows * nb, 256), 256, 0, s>>>(fmt, v.codes, v.scales, rows, nb,
                                                             static_cast<uint8_t*>(dst));
  }
  return launch_status();
}

qd_status qd_dequant(qd_fmt fmt, const void* packed, int64_t rows, int64_t cols, float* out, qd_stream_t stream) {
  if (!fmt_ok(fmt)) return QD_ERR_UNSUPPORTED;
  if (!packed || !out) return QD_ERR_INVALID_ARG;
  if (!shape_ok(fmt, rows, cols)) return QD_ERR_SHAPE;
  if (!aligned16(packed) || !aligned16(out)) return QD_ERR_ALIGN;
  k_dequant<<<grid_for(rows * cols, 256), 256, 0, (cudaStream_t)stream>>>(fmt, packed_view(fmt, packed, rows, cols),
                                                                          out);
  return launch_status();
}

qd_status qd_f16_to_f32(const uint16_t* in, float* out, int64_t n, qd_stream_t stream) {
  if (n < 0 || (n > 0 && (!in || !out))) return QD_ERR_INVALID_ARG;
  if (n == 0) return QD_OK;
  k_f16_to_f32<<<grid_for(n, 256), 256, 0, (cudaStream_t)stream>>>(in, out, n);
  return launch_status();
}

qd_status qd_bf16_to_f32(const uint16_t* in, float* out, int64_t n, qd_stream_t stream) {
  if (n < 0 || (n > 0 && (!in || !out))) return QD_ERR_INVALID_ARG;
  if (n == 0) return QD_OK;
  k_bf16_to_f32<<<grid_for(n, 256), 256, 0, (cudaStream_t)stream>>>(in, out, n);
  return launch_status();
}

}  // extern "C"
