// Load-time kernels: repack caller weights into the library's tiled HBM
// layouts (see msk_internal.h), validate E4M3 block scales, and the debug
// kernels (dequantise through the repacked layout; run the activation
// quantiser standalone).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "msk_device.cuh"
#include "msk_internal.h"

namespace msk {

// Dense: one thread per 16-byte output chunk.  With qk_rows > 0, rows of
// the first qk_rows (q and k heads) are permuted so that stored row 2i+0 is
// head row i and stored row 2i+1 is head row i + hd/2 (pairs of a rotation).
__global__ void repack_dense_kernel(const uint16_t* __restrict__ src, int64_t ld, int N, int K,
                                    uint8_t* __restrict__ dst, int qk_rows, int hd) {
  const int64_t nchunks = (int64_t)N * K / 8;
  const int kbs = K / 32;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < nchunks; q += (int64_t)gridDim.x * blockDim.x) {
    const int lane = (int)(q & 31);
    const int64_t blk = q >> 5;
    const int kb = (int)(blk % kbs);
    const int gi = (int)(blk / kbs);
    const int g = lane >> 2, c = lane & 3;
    int n = 8 * gi + g;
    if (n < qk_rows) {
      const int head = n / hd, j = n % hd;
      n = head * hd + ((j & 1) ? (j >> 1) + hd / 2 : (j >> 1));
    }
    const uint16_t* row = src + (int64_t)n * ld + 32 * kb;
    const int ks[8] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9, 16 + 2 * c, 17 + 2 * c, 24 + 2 * c, 25 + 2 * c};
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = (uint32_t)row[ks[2 * i]] | ((uint32_t)row[ks[2 * i + 1]] << 16);
    *reinterpret_cast<uint4*>(dst + q * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

struct Fp4Src {
  const uint8_t* packed;  // [rows][cols/2]
  const uint8_t* scales;  // [rows][cols/16]
};

__device__ __forceinline__ bool bad_scale(uint32_t b) { return (b & 0x80u) || ((b & 0x7Fu) == 0x7Fu); }

// Experts: one thread per (expert, matrix, 16-row tile, k128 chunk, lane).
// mat 0 = gate, 1 = up ([I][P]); mat 2 = down ([P][I]).  Lane L = 4 g + c
// writes its 32 code bytes; lanes 0..15 also write row L's 8 scales.
__global__ void repack_experts_kernel(const Fp4Src* __restrict__ srcs, int E, int P, int I, uint8_t* __restrict__ dst,
                                      int* __restrict__ bad) {
  const size_t eb = expert_bytes(P, I), g1b = expert_g1_bytes(P, I);
  const int u1 = g1_unit_bytes(P), u2 = g2_unit_bytes(I);
  const int64_t nt_gu = (int64_t)(I / 16) * (P / 128);  // tiles of gate (or up)
  const int64_t per_e = 2 * nt_gu + (int64_t)(P / 16) * (I / 128);
  const int64_t total = per_e * E * 32;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
    const int lane = (int)(q & 31);
    int64_t t = q >> 5;
    const int e = (int)(t / per_e);
    t %= per_e;
    int mat, rt, kc, cols;
    if (t < 2 * nt_gu) {
      mat = (int)(t / nt_gu);
      const int64_t r = t % nt_gu;
      rt = (int)(r / (P / 128));
      kc = (int)(r % (P / 128));
      cols = P;
    } else {
      mat = 2;
      const int64_t r = t - 2 * nt_gu;
      rt = (int)(r / (I / 128));
      kc = (int)(r % (I / 128));
      cols = I;
    }
    size_t off = (size_t)e * eb;
    if (mat < 2) off += (size_t)rt * u1 + g1_tile_off(kc, mat);
    else off += g1b + (size_t)(rt >> 1) * u2 + g2_tile_off(kc, rt & 1);
    const Fp4Src s = srcs[e * 3 + mat];
    const int g = lane >> 2, c = lane & 3;
    // this lane's 32 bytes: steps s = 0..7, registers j = 2 k8 + r8
    uint8_t out[32];
#pragma unroll
    for (int st = 0; st < 8; ++st)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int row = 16 * rt + g + 8 * (j & 1);
        const int col = 128 * kc + 16 * st + 8 * (j >> 1) + 2 * c;  // even: the pair's first element
        out[4 * st + j] = s.packed[(size_t)row * (cols / 2) + col / 2];
      }
    uint4 v0, v1;
    memcpy(&v0, out, 16);
    memcpy(&v1, out + 16, 16);
    *reinterpret_cast<uint4*>(dst + off + 16 * lane) = v0;
    *reinterpret_cast<uint4*>(dst + off + 512 + 16 * lane) = v1;
    if (lane < 16) {
      const uint8_t* sr = s.scales + (size_t)(16 * rt + lane) * (cols / 16) + kc * 8;
      uint8_t sc[8];
      int b = 0;
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        sc[st] = sr[st];
        b |= bad_scale(sc[st]);
      }
      uint2 sv;
      memcpy(&sv, sc, 8);
      *reinterpret_cast<uint2*>(dst + off + 1024 + lane * 8) = sv;
      if (b) atomicOr(bad, 1);
    }
  }
}

// Dequantise matrix `which` of expert `e` from the repacked layout.
__global__ void debug_dequant_kernel(const uint8_t* __restrict__ experts, const float* __restrict__ ts, int P, int I,
                                     int e, int which, float* __restrict__ out) {
  const int rows = which < 2 ? I : P, cols = which < 2 ? P : I;
  const size_t eb = expert_bytes(P, I), g1b = expert_g1_bytes(P, I);
  const float tscale = ts[3 * e + which];
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < (int64_t)rows * cols;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(q / cols), k = (int)(q % cols);
    const int rt = r >> 4, kc = k >> 7;
    size_t off = (size_t)e * eb;
    if (which < 2) off += (size_t)rt * g1_unit_bytes(P) + g1_tile_off(kc, which);
    else off += g1b + (size_t)(rt >> 1) * g2_unit_bytes(I) + g2_tile_off(kc, rt & 1);
    const uint8_t byte = experts[off + tile4_code_off(r & 15, k & 127)];
    const uint32_t code = (k & 1) ? (byte >> 4) : (byte & 0xF);
    const uint8_t sc = experts[off + tile4_scale_off(r & 15, k & 127)];
    const uint32_t h2 = e2m1x2_to_f16x2(code);
    const float ev = __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFF)));
    const float prod = ev * e4m3_to_f32(sc);  // exact
    out[q] = __fmul_rn(prod, tscale);
  }
}

// The kernel's activation quantiser on [rows][cols] fp32.
__global__ void debug_quantize_kernel(const float* __restrict__ x, int64_t nblocks, uint8_t* __restrict__ codes,
                                      uint8_t* __restrict__ scales) {
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblocks; b += (int64_t)gridDim.x * blockDim.x) {
    float v[16];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      v[j] = x[b * 16 + j];
      amax = fmaxf(amax, fabsf(v[j]));
    }
    uint32_t sc = 0;
    uint8_t out[16] = {0};
    if (amax > 0.f) {
      sc = f32_to_e4m3(amax / 6.0f);
      const float dec = e4m3_to_f32(sc);
      if (dec > 0.f) {
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const uint32_t byte = f32x2_to_e2m1x2(v[j] / dec, v[j + 1] / dec);
          out[j] = byte & 0xF;
          out[j + 1] = byte >> 4;
        }
      }
    }
    for (int j = 0; j < 16; ++j) codes[b * 16 + j] = out[j];
    scales[b] = (uint8_t)sc;
  }
}

cudaError_t repack_dense(const void* src, int64_t ld, int N, int K, void* dst, int qk_rows, int hd, cudaStream_t st) {
  const int64_t n = (int64_t)N * K / 8;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 4096);
  repack_dense_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint16_t*>(src), ld, N, K, static_cast<uint8_t*>(dst),
                                               qk_rows, hd);
  return cudaGetLastError();
}

cudaError_t repack_experts(const void* srcs_dev, int E, int P, int I, void* dst, int* bad_dev, cudaStream_t st) {
  const int64_t per_e = (int64_t)(I / 16) * (P / 128) * 2 + (int64_t)(P / 16) * (I / 128);
  const int64_t n = per_e * E * 32;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 8192);
  repack_experts_kernel<<<blocks, 256, 0, st>>>(static_cast<const Fp4Src*>(srcs_dev), E, P, I, static_cast<uint8_t*>(dst),
                                                bad_dev);
  return cudaGetLastError();
}

cudaError_t debug_dequant(const void* experts, const float* ts, int P, int I, int e, int which, float* out,
                          cudaStream_t st) {
  const int rows = which < 2 ? I : P, cols = which < 2 ? P : I;
  const int64_t n = (int64_t)rows * cols;
  debug_dequant_kernel<<<(int)std::min<int64_t>((n + 255) / 256, 4096), 256, 0, st>>>(
      static_cast<const uint8_t*>(experts), ts, P, I, e, which, out);
  return cudaGetLastError();
}

// Elementwise: the E2M1 code (low nibble of the packed pair) and the E4M3
// code of every value, through the same conversion helpers the kernels use.
__global__ void debug_convert_kernel(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ e2m1,
                                     uint8_t* __restrict__ e4m3) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float v = x[i];
    e2m1[i] = (uint8_t)(f32x2_to_e2m1x2(v, 0.f) & 0xFu);
    e4m3[i] = (uint8_t)f32_to_e4m3(v);
  }
}

cudaError_t debug_convert(const float* x, int64_t n, uint8_t* e2m1, uint8_t* e4m3, cudaStream_t st) {
  debug_convert_kernel<<<(int)std::min<int64_t>((n + 255) / 256, 8192), 256, 0, st>>>(x, n, e2m1, e4m3);
  return cudaGetLastError();
}

cudaError_t debug_quantize(const float* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* scales,
                           cudaStream_t st) {
  const int64_t nb = rows * cols / 16;
  debug_quantize_kernel<<<(int)std::min<int64_t>((nb + 255) / 256, 4096), 256, 0, st>>>(x, nb, codes, scales);
  return cudaGetLastError();
}

}  // namespace msk
