// One-GPU microbenchmarks behind the layer kernel's design.
//
// The pages report an instruction-cache probe (a 100 KB straight-line block
// alone against two such blocks run in sequence, and with a 20 KB partner)
// and single-GPU synchronisation costs (acquire polling, a fence when idle
// and with bulk copies in flight) ([orcarouter] "Su cosa vengono ancora
// spesi i 5,9 ms" and the icache / sync paragraphs of [newruntime]).  This
// program measures the same quantities on the local GPU, plus the streaming
// and staging paths the layer kernel uses (bulk-copy ring, per-warp stages,
// cp.async; activation staging from L2) and its grid barrier.  Every spin
// is bounded; a wait that runs out sets a flag that is printed.
//
// Output: one JSON object per line.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <vector>

#include "icache_bodies.cuh"

#define CK(x)                                                                         \
  do {                                                                                \
    cudaError_t e_ = (x);                                                             \
    if (e_ != cudaSuccess) {                                                          \
      printf("{\"error\": \"%s\", \"line\": %d}\n", cudaGetErrorString(e_), __LINE__); \
      return 1;                                                                       \
    }                                                                                 \
  } while (0)

namespace {

constexpr uint64_t kSpinLimit = 50000000ull;

__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mb_init(uint32_t b, uint32_t c) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(c) : "memory");
}
__device__ __forceinline__ void mb_expect(uint32_t b, uint32_t n) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(n) : "memory");
}
__device__ __forceinline__ void mb_arrive(uint32_t b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}
__device__ __forceinline__ bool mb_try(uint32_t b, uint32_t ph) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok)
               : "r"(b), "r"(ph)
               : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bulk(uint32_t d, const void* s, uint32_t n, uint32_t b) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(d),
               "l"(s), "r"(n), "r"(b)
               : "memory");
}
__device__ __forceinline__ void cp16(uint32_t d, const void* s) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(s) : "memory");
}
__device__ __forceinline__ uint32_t smem(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

extern __shared__ __align__(1024) uint8_t g_sm[];

__global__ void flush_l2(uint4* p, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = make_uint4((uint32_t)i, 1u, 2u, 3u);
}

// ---- synchronisation ------------------------------------------------------

// Blocks 0 and 1 bounce a counter through one word: block 0 waits for odd
// values and writes the next even one, block 1 the reverse (release stores,
// acquire polling).  One-way latency = elapsed / (2 n).
__global__ void pingpong(unsigned int* flag, int n, unsigned long long* out, int* fail) {
  if (threadIdx.x != 0 || blockIdx.x > 1) return;
  const unsigned int me = blockIdx.x;
  const uint64_t t0 = gtime();
  for (int i = 0; i < n; ++i) {
    const unsigned int want = 2u * i + me;
    uint64_t spins = 0;
    while (true) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
      if (v == want) break;
      if (++spins > kSpinLimit) {
        atomicExch(fail, 1);
        return;
      }
    }
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(want + 1u) : "memory");
  }
  if (me == 0) out[0] = gtime() - t0;
}

// Thread 0 times 64 gpu-scope fences (%globaltimer), first with nothing outstanding, then
// right after issuing 128 KB of bulk copies from HBM (not yet landed).
__global__ void fence_cost(const uint8_t* src, unsigned long long* out, int* fail) {
  const uint32_t bar = smem(g_sm) + 131072;
  if (threadIdx.x != 0) return;
  mb_init(bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  uint64_t c0 = gtime();
  for (int i = 0; i < 64; ++i) asm volatile("fence.acq_rel.gpu;" ::: "memory");
  uint64_t c1 = gtime();
  out[0] = c1 - c0;
  mb_expect(bar, 131072);
  for (int r = 0; r < 8; ++r) bulk(smem(g_sm) + r * 16384, src + (size_t)blockIdx.x * 131072 + r * 16384, 16384, bar);
  c0 = gtime();
  for (int i = 0; i < 64; ++i) asm volatile("fence.acq_rel.gpu;" ::: "memory");
  c1 = gtime();
  out[1] = c1 - c0;
  uint64_t spins = 0;
  while (!mb_try(bar, 0))
    if (++spins > kSpinLimit) {
      atomicExch(fail, 1);
      break;
    }
}

// The layer kernel's grid barrier: one 64-bit arrival counter that only
// grows; a block arrives with a release reduction and waits (acquire
// polling) for base + n * blocks.
__global__ void grid_barrier_loop(unsigned long long* cnt, int nb, unsigned long long* out, int* fail) {
  __shared__ int stop;
  unsigned long long base = 0;
  if (threadIdx.x == 0) {
    stop = 0;
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(cnt) : "memory");
    base = v - v % gridDim.x;
  }
  __syncthreads();
  const uint64_t t0 = gtime();
  for (int i = 1; i <= nb; ++i) {
    __syncthreads();
    if (threadIdx.x == 0 && !stop) {
      asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(cnt) : "memory");
      const unsigned long long target = base + (unsigned long long)i * gridDim.x;
      uint64_t spins = 0;
      while (true) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(cnt) : "memory");
        if ((long long)(v - target) >= 0) break;
        if (++spins > kSpinLimit) {
          atomicExch(fail, 1);
          stop = 1;
          break;
        }
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    out[2 * blockIdx.x] = t0;
    out[2 * blockIdx.x + 1] = gtime();
  }
}

// ---- streaming from HBM ---------------------------------------------------

// One producer thread (warp 8) fills a ring of ns slots of sb bytes with
// bulk copies; warps 0..7 wait on each slot, read it and release it.
__global__ void __launch_bounds__(288, 1) ring_stream(const uint8_t* src, size_t per_block, int ns, int sb,
                                                      float* sink, int* fail) {
  const uint8_t* s = src + (size_t)blockIdx.x * per_block;
  const uint32_t base = smem(g_sm), bars = base + 200 * 1024;
  if (threadIdx.x == 0) {
    for (int i = 0; i < ns; ++i) {
      mb_init(bars + 8 * i, 1);
      mb_init(bars + 8 * (32 + i), 8);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int ntiles = (int)(per_block / sb);
  if (threadIdx.x >= 256) {
    if (threadIdx.x == 256)
      for (int j = 0; j < ntiles; ++j) {
        const int slot = j % ns;
        if (j >= ns) {
          uint64_t spins = 0;
          while (!mb_try(bars + 8 * (32 + slot), ((j / ns) - 1) & 1))
            if (++spins > kSpinLimit) {
              atomicExch(fail, 1);
              return;
            }
        }
        mb_expect(bars + 8 * slot, sb);
        bulk(base + slot * sb, s + (size_t)j * sb, sb, bars + 8 * slot);
      }
    return;
  }
  float acc = 0.f;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = 0; j < ntiles; ++j) {
    const int slot = j % ns;
    uint64_t spins = 0;
    while (!mb_try(bars + 8 * slot, (j / ns) & 1))
      if (++spins > kSpinLimit) {
        atomicExch(fail, 1);
        break;
      }
    acc += *reinterpret_cast<const float*>(g_sm + slot * sb + ((w * 32 + lane) * 4) % sb);
    __syncwarp();
    if (lane == 0) mb_arrive(bars + 8 * (32 + slot));
  }
  if (acc == 1234.5f) sink[0] = acc;
}

// Eight warps, each streaming its own region through nst private stages of
// sb bytes (lane 0 issues one bulk copy per step), as the expert GEMMs do.
__global__ void __launch_bounds__(256, 1) warp_stream(const uint8_t* src, size_t per_warp, int nst, int sb,
                                                      float* sink, int* fail) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint8_t* s = src + ((size_t)blockIdx.x * 8 + w) * per_warp;
  const uint32_t base = smem(g_sm) + w * nst * sb, bars = smem(g_sm) + 216 * 1024 + w * 64;
  if (lane == 0)
    for (int i = 0; i < nst; ++i) mb_init(bars + 8 * i, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  const int nsteps = (int)(per_warp / sb);
  int issued = 0;
  for (; issued < nst - 1 && issued < nsteps; ++issued)
    if (lane == 0) {
      mb_expect(bars + 8 * (issued % nst), sb);
      bulk(base + (issued % nst) * sb, s + (size_t)issued * sb, sb, bars + 8 * (issued % nst));
    }
  float acc = 0.f;
  for (int j = 0; j < nsteps; ++j) {
    if (issued < nsteps) {
      if (lane == 0) {
        mb_expect(bars + 8 * (issued % nst), sb);
        bulk(base + (issued % nst) * sb, s + (size_t)issued * sb, sb, bars + 8 * (issued % nst));
      }
      ++issued;
    }
    uint64_t spins = 0;
    while (!mb_try(bars + 8 * (j % nst), (j / nst) & 1))
      if (++spins > kSpinLimit) {
        atomicExch(fail, 1);
        break;
      }
    acc += *reinterpret_cast<const float*>(g_sm + w * nst * sb + (j % nst) * sb + lane * 4);
    __syncwarp();
  }
  if (acc == 1234.5f) sink[0] = acc;
}

// All 256 threads stream with 16-byte cp.async, 12 groups of 8 KB in flight.
__global__ void __launch_bounds__(256, 1) cpasync_stream(const uint8_t* src, size_t per_block, float* sink) {
  constexpr int NS = 12;
  const uint8_t* s = src + (size_t)blockIdx.x * per_block;
  const uint32_t base = smem(g_sm);
  const int nch = (int)(per_block / 8192);
  float acc = 0.f;
  for (int j = 0; j < nch; ++j) {
    cp16(base + (j % NS) * 8192 + threadIdx.x * 16, s + (size_t)j * 8192 + threadIdx.x * 16);
    cp16(base + (j % NS) * 8192 + 4096 + threadIdx.x * 16, s + (size_t)j * 8192 + 4096 + threadIdx.x * 16);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group %0;" ::"n"(NS - 1) : "memory");
    acc += *reinterpret_cast<const float*>(g_sm + ((j + 1) % NS) * 8192 + threadIdx.x * 4);
  }
  if (acc == 1234.5f) sink[0] = acc;
}

// ---- activation staging ---------------------------------------------------

// Every block copies the same 16 x 8 KB rows (L2 resident) into padded rows:
// mode 0: 16-byte cp.async from all threads; mode 1: one bulk copy per row.
__global__ void __launch_bounds__(256, 1) stage_rows(const uint8_t* src, int mode, unsigned long long* out,
                                                     int* fail) {
  const uint32_t base = smem(g_sm), bar = base + 135168;
  if (threadIdx.x == 0) {
    mb_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const uint64_t t0 = gtime();
  if (mode == 0) {
    for (int i = threadIdx.x; i < 8192; i += 256) cp16(base + (i >> 9) * 8208 + (i & 511) * 16, src + i * 16);
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    if (threadIdx.x == 0) {
      mb_expect(bar, 131072);
      for (int r = 0; r < 16; ++r) bulk(base + r * 8208, src + r * 8192, 8192, bar);
    }
    uint64_t spins = 0;
    while (!mb_try(bar, 0))
      if (++spins > kSpinLimit) {
        atomicExch(fail, 1);
        break;
      }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    out[2 * blockIdx.x] = t0;
    out[2 * blockIdx.x + 1] = gtime();
  }
}

struct Body {
  int kb;
  void (*a)(float*, float, float);
  void (*b)(float*, float, float);
};
const Body kBodies[] = {ICACHE_TABLE};

float median(std::vector<float> v) {
  std::sort(v.begin(), v.end());
  return v[v.size() / 2];
}

}  // namespace

int main() {
  int nsm = 0;
  CK(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0));
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, 0));
  printf("{\"device\": \"%s\", \"sms\": %d, \"l2_bytes\": %d}\n", prop.name, nsm, prop.l2CacheSize);
  float* sink;
  CK(cudaMalloc(&sink, 4096));
  int* fail;
  CK(cudaMalloc(&fail, 4));
  CK(cudaMemset(fail, 0, 4));
  unsigned long long* tv;
  CK(cudaMalloc(&tv, 2 * 1024 * 8));
  std::vector<unsigned long long> h(2 * 1024);
  const size_t fl_n = (512ull << 20) / 16;
  uint4* fl;
  CK(cudaMalloc(&fl, fl_n * 16));
  cudaEvent_t e0, e1;
  CK(cudaEventCreate(&e0));
  CK(cudaEventCreate(&e1));
  auto time_launch = [&](void (*k)(float*, float, float)) {
    cudaEventRecord(e0);
    k<<<nsm, 256>>>(sink, 1.0001f, 0.5f);
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    return ms * 1000.f;
  };

  // ---- instruction cache: one block per SM executes N KB of straight-line
  // code once per thread
  const Body* partner = &kBodies[0];  // the 20 KB block
  for (const Body& b : kBodies) {
    std::vector<float> alone, pair, small, cold;
    for (int r = 0; r < 3; ++r) b.a<<<nsm, 256>>>(sink, 1.0001f, 0.5f);
    CK(cudaDeviceSynchronize());
    for (int r = 0; r < 15; ++r) alone.push_back(time_launch(b.a));
    for (int r = 0; r < 15; ++r) {
      b.b<<<nsm, 256>>>(sink, 1.0001f, 0.5f);  // another block of the same size in between
      pair.push_back(time_launch(b.a));
    }
    for (int r = 0; r < 15; ++r) {
      partner->b<<<nsm, 256>>>(sink, 1.0001f, 0.5f);  // a 20 KB block in between
      small.push_back(time_launch(b.a));
    }
    for (int r = 0; r < 7; ++r) {
      flush_l2<<<4 * nsm, 512>>>(fl, fl_n);
      cold.push_back(time_launch(b.a));
    }
    CK(cudaDeviceSynchronize());
    printf("{\"probe\": \"icache\", \"block_kb\": %d, \"alone_us\": %.2f, \"after_same_size_block_us\": %.2f, "
           "\"after_20kb_block_us\": %.2f, \"after_l2_flush_us\": %.2f}\n",
           b.kb, median(alone), median(pair), median(small), median(cold));
  }

  // ---- synchronisation
  unsigned int* flag;
  CK(cudaMalloc(&flag, 256));
  {
    std::vector<float> v;
    for (int r = 0; r < 5; ++r) {
      CK(cudaMemset(flag, 0, 256));
      pingpong<<<2, 32>>>(flag, 1000, tv, fail);
      CK(cudaDeviceSynchronize());
      CK(cudaMemcpy(h.data(), tv, 8, cudaMemcpyDeviceToHost));
      v.push_back((float)h[0] / 2000.f);
    }
    printf("{\"probe\": \"acquire_poll_one_way\", \"ns\": %.1f}\n", median(v));
  }
  const size_t per_block = 4ull << 20;
  uint8_t* big;
  CK(cudaMalloc(&big, per_block * nsm));
  CK(cudaMemset(big, 1, per_block * nsm));
  CK(cudaFuncSetAttribute(fence_cost, cudaFuncAttributeMaxDynamicSharedMemorySize, 136 * 1024));
  {
    std::vector<float> idle, busy;
    for (int r = 0; r < 5; ++r) {
      flush_l2<<<4 * nsm, 512>>>(fl, fl_n);
      fence_cost<<<1, 32, 136 * 1024>>>(big, tv, fail);
      CK(cudaDeviceSynchronize());
      CK(cudaMemcpy(h.data(), tv, 16, cudaMemcpyDeviceToHost));
      idle.push_back((float)h[0] / 64.f);
      busy.push_back((float)h[1] / 64.f);
    }
    printf("{\"probe\": \"fence_acq_rel_gpu\", \"idle_ns\": %.1f, \"with_128kb_bulk_in_flight_ns\": %.1f}\n",
           median(idle), median(busy));
  }
  {
    unsigned long long* cnt;
    CK(cudaMalloc(&cnt, 64));
    CK(cudaMemset(cnt, 0, 64));
    std::vector<float> v;
    for (int r = 0; r < 5; ++r) {
      int nb = 200;
      void* args[] = {&cnt, &nb, &tv, &fail};
      CK(cudaLaunchCooperativeKernel((void*)grid_barrier_loop, nsm, 256, args, 0, 0));
      CK(cudaDeviceSynchronize());
      CK(cudaMemcpy(h.data(), tv, 2 * nsm * 8, cudaMemcpyDeviceToHost));
      unsigned long long mn = ~0ull, mx = 0;
      for (int b = 0; b < nsm; ++b) {
        mn = std::min(mn, h[2 * b]);
        mx = std::max(mx, h[2 * b + 1]);
      }
      v.push_back((float)(mx - mn) / 1000.f / nb);
    }
    printf("{\"probe\": \"grid_barrier\", \"blocks\": %d, \"us_per_barrier\": %.3f}\n", nsm, median(v));
  }

  // ---- streaming from HBM into shared memory (every block its own region)
  const double total = (double)per_block * nsm;
  auto bw = [&](float ms) { return total / (ms * 1e-3) / 1e9; };
  CK(cudaFuncSetAttribute(ring_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, 208 * 1024));
  CK(cudaFuncSetAttribute(warp_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024));
  CK(cudaFuncSetAttribute(cpasync_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, 208 * 1024));
  struct RingCfg {
    int ns, sb;
  };
  for (RingCfg c : {RingCfg{5, 16384}, RingCfg{4, 4608}, RingCfg{16, 4608}}) {
    std::vector<float> t;
    for (int r = 0; r < 5; ++r) {
      cudaEventRecord(e0);
      ring_stream<<<nsm, 288, 208 * 1024>>>(big, per_block, c.ns, c.sb, sink, fail);
      cudaEventRecord(e1);
      CK(cudaEventSynchronize(e1));
      float ms;
      cudaEventElapsedTime(&ms, e0, e1);
      t.push_back(ms);
    }
    printf("{\"probe\": \"stream_ring_one_producer\", \"slots\": %d, \"slot_bytes\": %d, \"GBps\": %.0f}\n", c.ns,
           c.sb, bw(median(t)));
  }
  for (RingCfg c : {RingCfg{4, 4608}, RingCfg{2, 9216}}) {
    std::vector<float> t;
    for (int r = 0; r < 5; ++r) {
      cudaEventRecord(e0);
      warp_stream<<<nsm, 256, 220 * 1024>>>(big, per_block / 8, c.ns, c.sb, sink, fail);
      cudaEventRecord(e1);
      CK(cudaEventSynchronize(e1));
      float ms;
      cudaEventElapsedTime(&ms, e0, e1);
      t.push_back(ms);
    }
    printf("{\"probe\": \"stream_per_warp_stages\", \"stages\": %d, \"stage_bytes\": %d, \"GBps\": %.0f}\n", c.ns,
           c.sb, bw(median(t)));
  }
  {
    std::vector<float> t;
    for (int r = 0; r < 5; ++r) {
      cudaEventRecord(e0);
      cpasync_stream<<<nsm, 256, 208 * 1024>>>(big, per_block, sink);
      cudaEventRecord(e1);
      CK(cudaEventSynchronize(e1));
      float ms;
      cudaEventElapsedTime(&ms, e0, e1);
      t.push_back(ms);
    }
    printf("{\"probe\": \"stream_cp_async_16B\", \"inflight_kb\": 96, \"GBps\": %.0f}\n", bw(median(t)));
  }

  // ---- activation staging: 128 KB shared by every block, from L2
  CK(cudaFuncSetAttribute(stage_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, 136 * 1024));
  for (int mode = 0; mode < 2; ++mode) {
    std::vector<float> span;
    for (int r = 0; r < 7; ++r) {
      CK(cudaMemset(big, r, 131072));
      stage_rows<<<nsm, 256, 136 * 1024>>>(big, mode, tv, fail);
      CK(cudaDeviceSynchronize());
      CK(cudaMemcpy(h.data(), tv, 2 * nsm * 8, cudaMemcpyDeviceToHost));
      unsigned long long mn = ~0ull, mx = 0;
      for (int b = 0; b < nsm; ++b) {
        mn = std::min(mn, h[2 * b]);
        mx = std::max(mx, h[2 * b + 1]);
      }
      span.push_back((float)(mx - mn) / 1000.f);
    }
    printf("{\"probe\": \"stage_128kb_shared_rows\", \"method\": \"%s\", \"us\": %.2f}\n",
           mode ? "bulk copy per row" : "cp.async 16 B", median(span));
  }
  int hf = 0;
  CK(cudaMemcpy(&hf, fail, 4, cudaMemcpyDeviceToHost));
  printf("{\"probe\": \"bounded_waits\", \"any_ran_out\": %d}\n", hf);
  return 0;
}
