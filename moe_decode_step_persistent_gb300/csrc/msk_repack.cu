// Load-time kernels: repack caller weights into the library's tiled HBM
// layouts (see msk_internal.h), validate E4M3 block scales, and the debug
// kernels (dequantise through the repacked layout; run the activation
// quantiser standalone).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "msk_device.cuh"
#include "msk_internal.h"
#include "msk_tc.cuh"

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

// Experts: one thread per (expert, matrix, row, 32-element chunk of K): its
// 16 code bytes go to their core-matrix row in the tensor-core layout (one
// 16-byte store), its two block scales to their scale chunk; any scale with
// the sign bit set or the NaN code raises *bad.  mat 0 = gate, 1 = up
// ([I][P]); mat 2 = down ([P][I]).
__global__ void repack_experts_kernel(const Fp4Src* __restrict__ srcs, int E, int P, int I, uint8_t* __restrict__ dst,
                                      int* __restrict__ bad) {
  const size_t eb = xexpert_bytes(P, I);
  const int64_t n_gu = (int64_t)I * (P / 32);  // chunks of gate (or up)
  const int64_t per_e = 2 * n_gu + (int64_t)P * (I / 32);
  const int64_t total = per_e * E;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(q / per_e);
    int64_t t = q % per_e;
    int mat, cols;
    if (t < 2 * n_gu) {
      mat = (int)(t / n_gu);
      t %= n_gu;
      cols = P;
    } else {
      mat = 2;
      t -= 2 * n_gu;
      cols = I;
    }
    const int r = (int)(t / (cols / 32)), k = 32 * (int)(t % (cols / 32));
    const Fp4Src s = srcs[e * 3 + mat];
    uint8_t* de = dst + (size_t)e * eb;
    *reinterpret_cast<uint4*>(de + xcode_off(P, I, mat, r, k)) =
        *reinterpret_cast<const uint4*>(s.packed + (size_t)r * (cols / 2) + k / 2);
    const uint8_t s0 = s.scales[(size_t)r * (cols / 16) + k / 16], s1 = s.scales[(size_t)r * (cols / 16) + k / 16 + 1];
    de[xscale_off(P, I, mat, r, k)] = s0;
    de[xscale_off(P, I, mat, r, k + 16)] = s1;
    if (bad_scale(s0) || bad_scale(s1)) atomicOr(bad, 1);
  }
}

// Dequantise matrix `which` of expert `e` from the repacked layout.
__global__ void debug_dequant_kernel(const uint8_t* __restrict__ experts, const float* __restrict__ ts, int P, int I,
                                     int e, int which, float* __restrict__ out) {
  const int rows = which < 2 ? I : P, cols = which < 2 ? P : I;
  const uint8_t* ex = experts + (size_t)e * xexpert_bytes(P, I);
  const float tscale = ts[3 * e + which];
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < (int64_t)rows * cols;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(q / cols), k = (int)(q % cols);
    const uint8_t byte = ex[xcode_off(P, I, which, r, k)];
    const uint32_t code = (k & 1) ? (byte >> 4) : (byte & 0xF);
    const uint8_t sc = ex[xscale_off(P, I, which, r, k)];
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
  const int64_t n = ((int64_t)2 * I * (P / 32) + (int64_t)P * (I / 32)) * E;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 16384);
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

// ---------------------------------------------------------------------------
// One block-scaled NVFP4 tile on the tensor cores, for tests: D[128][16] =
// A[128][K] B[n][K]^T (rows of B past n are zero), A and B given in the
// natural layout ([rows][K/2] codes, element 2i in the low nibble of byte
// i; [rows][K/16] E4M3 scales).  The operand images are built in shared
// memory with the same layout helpers as the expert repack and the layer
// kernel, then multiplied by the same tcgen05 sequence: per MMA, the A and
// B scale chunks into tensor memory, then kind::mxf4nvf4 into one fp32
// accumulator, committed to an mbarrier; four warps read the accumulator.
// One block of 128 threads.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int fp4_tile_smem(int K) {
  return ((K + kUStageK - 1) / kUStageK) * kUStageBytes + kUN * K / 2 + (K / 64) * 512;
}

__global__ void __launch_bounds__(128, 1) debug_fp4_tile_kernel(const uint8_t* __restrict__ ac,
                                                               const uint8_t* __restrict__ as,
                                                               const uint8_t* __restrict__ bc,
                                                               const uint8_t* __restrict__ bs, int nb, int K,
                                                               float* __restrict__ d, uint32_t* __restrict__ err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_bar;
  __shared__ int s_zero;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nst = (K + kUStageK - 1) / kUStageK, kc = K / 32, kb = K / 16;
  uint8_t* A = sm;
  uint8_t* B = sm + nst * kUStageBytes;
  uint8_t* Bsf = B + kUN * K / 2;
  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    s_zero = 0;
    mbar_init(smem_u32(&s_bar), 1);
    mbar_fence_init();
  }
  for (int i = tid; i < kURows * kc; i += blockDim.x) {
    const int m = i / kc, k = 32 * (i % kc);
    *reinterpret_cast<uint4*>(A + (k / kUStageK) * kUStageBytes + umma_code_off(kURows, m, k % kUStageK)) =
        *reinterpret_cast<const uint4*>(ac + (size_t)m * (K / 2) + k / 2);
  }
  for (int i = tid; i < kURows * kb; i += blockDim.x) {
    const int m = i / kb, b = i % kb, s = b / (kUStageK / 16);
    A[s * kUStageBytes + 64 * ustage_k(K, s) + umma_sf_off(m, b % (kUStageK / 16))] = as[(size_t)m * kb + b];
  }
  for (int i = tid; i < kUN * kc; i += blockDim.x) {
    const int n = i / kc, k = 32 * (i % kc);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < nb) v = *reinterpret_cast<const uint4*>(bc + (size_t)n * (K / 2) + k / 2);
    *reinterpret_cast<uint4*>(B + umma_code_off(kUN, n, k)) = v;
  }
  for (int i = tid; i < (K / 64) * 32; i += blockDim.x) *reinterpret_cast<uint4*>(Bsf + 16 * i) = make_uint4(0, 0, 0, 0);
  __syncthreads();
  for (int i = tid; i < nb * kb; i += blockDim.x) {
    const int n = i / kb, b = i % kb;
    Bsf[umma_sf_off(n, b)] = bs[(size_t)n * kb + b];
  }
  fence_proxy_async_shared();  // the images (generic-proxy writes) before the tensor core reads them
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s_tmem;
  if (tid == 0) {
    const uint32_t idesc = idesc_mxf4nvf4(kUN);
    int j = 0;
    for (int s = 0; s < nst; ++s) {
      const int kst = ustage_k(K, s);
      const uint32_t sa = smem_u32(A + s * kUStageBytes);
      for (int kk = 0; kk < kst / 64; ++kk, ++j) {
        tc_cp_sf(tb + 64 + 4 * j, umma_desc(sa + 64 * kst + 512 * kk, 128, 128));
        tc_cp_sf(tb + 256 + 4 * j, umma_desc(smem_u32(Bsf) + 512 * j, 128, 128));
        mma_mxf4nvf4(tb, umma_desc(sa + 4096 * kk, 16 * kURows, 128), umma_desc(smem_u32(B) + 512 * j, 16 * kUN, 128),
                     idesc, tb + 64 + 4 * j, tb + 256 + 4 * j, j > 0);
      }
    }
    tc_commit(smem_u32(&s_bar));
  }
  const bool ok = mbar_wait(smem_u32(&s_bar), 0, gtimer() + 1000000000ull, &s_zero);
  tc_fence_after();
  if (ok) {
    float v[16];
    tmem_ld16(tmem_lane_addr(tb, 32 * warp, 0), v);
#pragma unroll
    for (int i = 0; i < 16; ++i) d[(32 * warp + lane) * kUN + i] = v[i];
  } else if (lane == 0) {
    atomicOr(err, 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t debug_fp4_tile(const uint8_t* ac, const uint8_t* as, const uint8_t* bc, const uint8_t* bs, int nb, int K,
                           float* d, uint32_t* err, cudaStream_t st) {
  const int smem = fp4_tile_smem(K);
  cudaError_t e = cudaFuncSetAttribute(debug_fp4_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  debug_fp4_tile_kernel<<<1, 128, smem, st>>>(ac, as, bc, bs, nb, K, d, err);
  return cudaGetLastError();
}

}  // namespace msk
