// msk_attention_noalloc: the split-KV GQA attention of the layer kernel as a
// standalone call that performs no device allocation.
//
// Why it exists: some callers cannot call cudaMalloc at the point where they
// need attention -- code running inside a serving framework that hands out
// all device memory from its own pre-sized pool, or code that must not
// allocate while the framework is recording work for later replay.  The
// model-based entry points allocate their scratch in msk_create; this one
// keeps its scratch (the per-block attention partials and the grid barrier
// words) in one file-scope device array instead.
//
// The array is a fixed kNoAllocScratchBytes (6 MiB) on every GPU that loads
// the library, held until the process exits.  Every call shares it and it
// keeps the previous call's contents, so calls whose executions overlap on
// the GPU (two streams, two host threads) race: serialise them.  The
// barrier and error words are cleared at the start of every call; the
// partials need no clearing (each is written before it is read).  The call
// waits for its stream to finish (to read the error word), so it cannot be
// recorded into a stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/msk.h"
#include "msk_phases_dense.cuh"

namespace msk {

constexpr size_t kNoAllocScratchBytes = 6u << 20;
constexpr size_t kNoAllocHeader = 512;  // [0,256) barrier words, [256,512) error words

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

template <int HD>
__global__ void __launch_bounds__(kConsThreads, 1) msk_attention_noalloc_kernel(const __grid_constant__ LaunchArgs args) {
  stage_args(args);
  Ctx c;
  c.seq = 0;
  c.nbar = 0;
  c.xseq = 0;
  c.xunit = 0;
  c.nstg = 0;
  c.sg = 0;
  c.bar0 = threadIdx.x == 0 ? grid_barrier_base(args.s.bar) : 0ull;  // (the shared copy is not yet complete)
  if (c.tid() == 0) {
    c.misc()->abort = 0;
    c.misc()->zero = 0;
    c.misc()->spare = 0;
    mbar_init(c.bar(BAR_STG), 1);  // the attention phase stages its queries with it
    for (int i = 0; i < kAttnStages; ++i) mbar_init(c.bar(BAR_KV + i), 1);  // ... and its keys and values
    c.misc()->kvmap = reinterpret_cast<unsigned long long>(&args.kv_map);
    prefetch_tensormap(&args.kv_map);
    mbar_fence_init();
  }
  __syncthreads();
  attention_phase<HD>(c);
  if (!grid_barrier(c, PH_ATTN)) return;
  combine_phase<HD>(c);
}

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device
bool g_ready[kMaxDevices] = {};
std::mutex g_setup_mutex;  // first calls from several host threads run the set-up once

// One-time set-up on the current device: the device address of the static
// scratch array (its host-side name is only a stand-in) and the kernels'
// shared-memory opt-in.  No allocation.  Serialised by g_setup_mutex; a
// failed set-up is retried by the next call.
cudaError_t setup_device(int dev) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_ready[dev]) return cudaSuccess;
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(msk_attention_noalloc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(msk_attention_noalloc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  g_scratch_ptr[dev] = p;
  g_ready[dev] = true;
  return cudaSuccess;
}

}  // namespace
}  // namespace msk

using namespace msk;

extern "C" msk_status msk_attention_noalloc(const void* q, const void* kv_layer, int32_t tokens, int32_t n_q_heads,
                                            int32_t n_kv_heads, int32_t head_dim, int32_t max_seq, int32_t pos0,
                                            int32_t window, void* out, void* stream) {
  if (q == nullptr || kv_layer == nullptr || out == nullptr) return MSK_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return MSK_ERR_SHAPE;
  if (tokens <= 0 || tokens > kMaxT || n_kv_heads <= 0 || n_q_heads <= 0 || n_q_heads % n_kv_heads) return MSK_ERR_SHAPE;
  if ((n_q_heads / n_kv_heads) * tokens > 64) return MSK_ERR_SHAPE;
  if (n_q_heads * head_dim > kMaxK) return MSK_ERR_SHAPE;
  if (window < 0 || pos0 < 0 || max_seq <= 0 || pos0 + tokens > max_seq) return MSK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_layer) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return MSK_ERR_ALIGNMENT;
  int dev = 0, nsm = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MSK_ERR_CUDA;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MSK_ERR_CUDA;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
    return MSK_ERR_UNSUPPORTED_DEVICE;
  // every kv head needs at least one block of the grid (one per SM): the
  // attention stage gives each head nsm / n_kv_heads key splits, and the
  // combine reads one partial per split of every head
  if (n_kv_heads > nsm) return MSK_ERR_SHAPE;
  // the scratch this call needs must fit the fixed array
  const size_t need = kNoAllocHeader + (size_t)nsm * 64 * 2 * 4 + (size_t)nsm * 64 * head_dim * 4;
  if (need > kNoAllocScratchBytes) return MSK_ERR_SHAPE;
  if (setup_device(dev) != cudaSuccess) return MSK_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(g_scratch_ptr[dev]);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  LaunchArgs a{};
  a.dm.Hq = n_q_heads;
  a.dm.Hkv = n_kv_heads;
  a.dm.hd = head_dim;
  a.dm.T = tokens;
  a.dm.max_seq = max_seq;
  a.dm.nctas = nsm;
  a.cur.window = window;
  a.s.q_stash = const_cast<uint16_t*>(static_cast<const uint16_t*>(q));
  a.s.attn_o = static_cast<uint16_t*>(out);
  a.s.bar = reinterpret_cast<unsigned long long*>(base);
  a.s.err = reinterpret_cast<uint32_t*>(base + 256);
  a.s.ml_part = reinterpret_cast<float*>(base + kNoAllocHeader);
  a.s.o_part = reinterpret_cast<float*>(base + kNoAllocHeader + (size_t)nsm * 64 * 2 * 4);
  a.kv_cur = const_cast<uint16_t*>(static_cast<const uint16_t*>(kv_layer));
  a.kv_z0 = 0;
  if (!encode_kv_map(&a.kv_map, kv_layer, head_dim, max_seq, 2LL * n_kv_heads)) return MSK_ERR_CUDA;
  a.pos0 = pos0;
  tree_masks(nullptr, tokens, window, a.depth, a.vis);  // the chain
  a.budget_ns = 200ull * 1000 * 1000;
  a.inject_bar = -1;
  a.inject_cta = -1;

  if (cudaMemsetAsync(base, 0, kNoAllocHeader, st) != cudaSuccess) return MSK_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nsm);
  cfg.blockDim = dim3(kConsThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = head_dim == 128 ? cudaLaunchKernelEx(&cfg, msk_attention_noalloc_kernel<128>, a)
                                         : cudaLaunchKernelEx(&cfg, msk_attention_noalloc_kernel<64>, a);
  if (le != cudaSuccess) return MSK_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MSK_ERR_CUDA;
  uint32_t err = 0;
  if (cudaMemcpy(&err, base + 256, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) return MSK_ERR_CUDA;
  return err ? MSK_ERR_TIMEOUT : MSK_OK;
}
