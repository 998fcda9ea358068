// C ABI of libmsk.so (declared in include/msk.h): model creation, weight
// loading (validation + repack into library layouts), the per-layer launch
// loop, error readback and test hooks.  Host code only; every step of the
// verify computation runs in the kernels of msk_layer.cu.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/msk.h"
#include "msk_internal.h"

namespace msk {
cudaError_t launch_layer(const LaunchArgs& args, bool timing, bool chained, cudaStream_t st);
cudaError_t prepare_launch();
int smem_bytes();
cudaError_t repack_dense(const void* src, int64_t ld, int N, int K, void* dst, int qk_rows, int hd, cudaStream_t st);
cudaError_t repack_experts(const void* srcs_dev, int E, int P, int I, void* dst, int* bad_dev, cudaStream_t st);
cudaError_t debug_dequant(const void* experts, const float* ts, int P, int I, int e, int which, float* out,
                          cudaStream_t st);
cudaError_t debug_convert(const float* x, int64_t n, uint8_t* e2m1, uint8_t* e4m3, cudaStream_t st);
cudaError_t debug_quantize(const float* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* scales,
                           cudaStream_t st);
cudaError_t debug_fp4_tile(const uint8_t* ac, const uint8_t* as, const uint8_t* bc, const uint8_t* bs, int nb, int K,
                           float* d, uint32_t* err, cudaStream_t st);
}  // namespace msk

using namespace msk;

namespace {

constexpr uint64_t kDefaultBudgetNs = 200ull * 1000 * 1000;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct LayerAlloc {
  void* base = nullptr;
  size_t bytes = 0;
};

}  // namespace

struct msk_model {
  msk_model_config cfg{};
  std::vector<uint8_t> is_global;
  Dims dm{};
  int device = 0;
  std::vector<LayerDev> layers;
  std::vector<LayerAlloc> allocs;
  Scratch s{};
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  size_t weight_bytes = 0;
  bool timing = false;
  unsigned long long* timeline = nullptr;  // [n_layers][nctas][slots]
  int last_launches = 0;
  int last_first = 0;  // layer of the most recent call's first launch
  uint64_t budget = kDefaultBudgetNs;
  int inject_bar = -1, inject_cta = -1;
  int kv_prefetch_rows = 2048;  // cap on the next layer's cached KV rows prefetched into L2
  bool launch_timing = false;
  std::vector<cudaEvent_t> ev;  // [2 * n_layers]
  // the captured step (msk_step_graph_capture / msk_step_graph_launch)
  StepInfo* step_dev = nullptr;   // device record the replayed launches read
  StepInfo* step_host = nullptr;  // pinned staging copy of it
  cudaStream_t cap_stream = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t graph_exec = nullptr;
  // the KV cache's tiled-copy map, encoded for the cache last passed in
  const void* kv_map_base = nullptr;
  CUtensorMap kv_map{};
};

#define MSK_CUDA(x)                             \
  do {                                          \
    cudaError_t e_ = (x);                       \
    if (e_ != cudaSuccess) return MSK_ERR_CUDA; \
  } while (0)

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

namespace msk {

// cuTensorMapEncodeTiled from the driver, looked up once through the
// runtime (the library does not link the driver library itself).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_kv_map(CUtensorMap* map, const void* kv, int hd, int max_seq, long long planes) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr || hd % 64 != 0 || max_seq <= 0 || planes <= 0) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)max_seq, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)hd * 2, (cuuint64_t)hd * 2 * (cuuint64_t)max_seq};
  const cuuint32_t box[3] = {64, (cuuint32_t)kAttnChunk, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kv), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace msk

// The model's KV map for `kv` (re-encoded when the cache changes).
static bool prepare_kv_map(msk_model* m, const void* kv) {
  if (m->kv_map_base == kv) return true;
  const Dims& d = m->dm;
  if (!msk::encode_kv_map(&m->kv_map, kv, d.hd, d.max_seq, (long long)d.n_layers * 2 * d.Hkv)) {
    m->kv_map_base = nullptr;
    return false;
  }
  m->kv_map_base = kv;
  return true;
}

extern "C" const char* msk_status_string(msk_status s) {
  switch (s) {
    case MSK_OK: return "ok";
    case MSK_ERR_INVALID_ARG: return "invalid argument";
    case MSK_ERR_SHAPE: return "unsupported or inconsistent shape";
    case MSK_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case MSK_ERR_BAD_SCALE: return "E4M3 block scale is NaN or negative";
    case MSK_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103 (GB300)";
    case MSK_ERR_OOM: return "out of device memory";
    case MSK_ERR_CUDA: return "CUDA runtime error";
    case MSK_ERR_TIMEOUT: return "device wait exceeded its time budget";
    case MSK_ERR_NOT_LOADED: return "layer weights not loaded";
  }
  return "unknown status";
}

extern "C" msk_status msk_create(const msk_model_config* cfg, msk_model** out) {
  if (out == nullptr || cfg == nullptr) return MSK_ERR_INVALID_ARG;
  *out = nullptr;
  const msk_model_config& c = *cfg;
  if (c.n_layers <= 0 || c.layer_is_global == nullptr) return MSK_ERR_INVALID_ARG;
  if (c.hidden <= 0 || c.hidden % 128 || c.hidden > kMaxK) return MSK_ERR_SHAPE;
  if (c.pooled <= 0 || c.pooled % 128 || c.pooled > 2048) return MSK_ERR_SHAPE;
  if (c.inter <= 0 || c.inter % 128 || c.inter > 2048) return MSK_ERR_SHAPE;
  if (c.head_dim != 64 && c.head_dim != 128) return MSK_ERR_SHAPE;
  if (c.n_kv_heads <= 0 || c.n_q_heads <= 0 || c.n_q_heads % c.n_kv_heads) return MSK_ERR_SHAPE;
  if (c.n_q_heads * c.head_dim > kMaxK) return MSK_ERR_SHAPE;
  if (c.verify_tokens <= 0 || c.verify_tokens > kMaxT) return MSK_ERR_SHAPE;
  if ((c.n_q_heads / c.n_kv_heads) * c.verify_tokens > 64) return MSK_ERR_SHAPE;
  if (c.top_k <= 0 || c.top_k > 8 || c.n_experts < c.top_k || c.n_experts > 256 || c.n_experts % 8)
    return MSK_ERR_SHAPE;
  if (c.max_seq < c.verify_tokens || c.window < 0) return MSK_ERR_SHAPE;
  if (c.prefetch_experts < 0 || c.prefetch_experts > 32) return MSK_ERR_INVALID_ARG;

  int dev = 0;
  MSK_CUDA(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  MSK_CUDA(cudaGetDeviceProperties(&prop, dev));
  if (!(prop.major == 10 && prop.minor == 3)) return MSK_ERR_UNSUPPORTED_DEVICE;
  int coop = 0;
  MSK_CUDA(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev));
  int optin = 0;
  MSK_CUDA(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
  if (!coop || optin < smem_bytes()) return MSK_ERR_UNSUPPORTED_DEVICE;

  msk_model* m = new (std::nothrow) msk_model();
  if (m == nullptr) return MSK_ERR_OOM;
  m->cfg = c;
  m->is_global.assign(c.layer_is_global, c.layer_is_global + c.n_layers);
  m->cfg.layer_is_global = nullptr;
  m->device = dev;
  Dims& d = m->dm;
  d.D = c.hidden;
  d.Hq = c.n_q_heads;
  d.Hkv = c.n_kv_heads;
  d.hd = c.head_dim;
  d.P = c.pooled;
  d.E = c.n_experts;
  d.topk = c.top_k;
  d.I = c.inter;
  d.T = c.verify_tokens;
  d.max_seq = c.max_seq;
  d.n_layers = c.n_layers;
  d.pf_experts = c.prefetch_experts;
  d.nctas = prop.multiProcessorCount;
  d.eps = c.rms_eps;
  d.theta = c.rope_theta;
  if (c.wait_budget_ns) m->budget = c.wait_budget_ns;
  m->layers.assign(c.n_layers, LayerDev{});
  m->allocs.assign(c.n_layers, LayerAlloc{});
  for (int l = 0; l < c.n_layers; ++l) m->layers[l].window = m->is_global[l] ? 0 : c.window;

  // scratch
  const int T = d.T, NC = d.nctas;
  const size_t sizes[] = {
      (size_t)T * d.Hq * d.hd * 2,      // q_stash
      (size_t)NC * 64 * d.hd * 4,       // o_part
      (size_t)NC * 64 * 2 * 4,          // ml_part
      (size_t)T * d.Hq * d.hd * 2,      // attn_o
      (size_t)T * d.D * 2,              // h1
      (size_t)T * d.P * 2,              // pooled
      (size_t)T * d.E * 4,              // logits
      (size_t)T * d.topk * (d.I / 2),   // sq_codes
      (size_t)T * d.topk * (d.I / 16),  // sq_scales
      (size_t)T * d.topk * d.P * 2,     // y
      (size_t)T * d.P * 2,              // mvec
      (size_t)T * (d.hd / 2) * 2 * 4,   // rope
      64,                               // bar
      64,                               // err
      (size_t)(d.hd / 2) * 8,           // inv_freq
      (size_t)(2 * d.E + 2) * 4,        // x1_done, xq
      (size_t)T * d.P / 2,              // x4_codes
      (size_t)NC * kMaxT * 4,           // ss_part
      (size_t)T * d.P / 16,             // x4_scales
      33 * 4,                           // pf_out
  };
  const int nbuf = sizeof(sizes) / sizeof(sizes[0]);
  size_t total = 0;
  for (int i = 0; i < nbuf; ++i) total += align_up(sizes[i], 256);
  if (cudaMalloc(&m->scratch, total) != cudaSuccess) {
    delete m;
    return MSK_ERR_OOM;
  }
  m->scratch_bytes = total;
  uint8_t* p = static_cast<uint8_t*>(m->scratch);
  void* ptrs[24];
  for (int i = 0; i < nbuf; ++i) {
    ptrs[i] = p;
    p += align_up(sizes[i], 256);
  }
  m->s.q_stash = (uint16_t*)ptrs[0];
  m->s.o_part = (float*)ptrs[1];
  m->s.ml_part = (float*)ptrs[2];
  m->s.attn_o = (uint16_t*)ptrs[3];
  m->s.h1 = (uint16_t*)ptrs[4];
  m->s.pooled = (uint16_t*)ptrs[5];
  m->s.logits = (float*)ptrs[6];
  m->s.sq_codes = (uint8_t*)ptrs[7];
  m->s.sq_scales = (uint8_t*)ptrs[8];
  m->s.y = (uint16_t*)ptrs[9];
  m->s.mvec = (uint16_t*)ptrs[10];
  m->s.rope = (float*)ptrs[11];
  m->s.bar = (unsigned long long*)ptrs[12];
  m->s.err = (uint32_t*)ptrs[13];
  m->s.inv_freq = (const double*)ptrs[14];
  m->s.x1_done = (uint32_t*)ptrs[15];
  m->s.xq = m->s.x1_done + d.E;
  m->s.x4_codes = (uint8_t*)ptrs[16];
  m->s.ss_part = (float*)ptrs[17];
  m->s.x4_scales = (uint8_t*)ptrs[18];
  m->s.pf_out = (int*)ptrs[19];
  // RoPE inverse frequencies theta^(-2i/d), i < d/2 (a model constant)
  std::vector<double> inv_freq(d.hd / 2);
  for (int i = 0; i < d.hd / 2; ++i) inv_freq[i] = std::pow((double)d.theta, -2.0 * i / d.hd);
  if (cudaMemset(m->scratch, 0, total) != cudaSuccess ||
      cudaMemcpy(ptrs[14], inv_freq.data(), inv_freq.size() * 8, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(m->scratch);
    delete m;
    return MSK_ERR_CUDA;
  }
  *out = m;
  return MSK_OK;
}

extern "C" void msk_destroy(msk_model* m) {
  if (m == nullptr) return;
  for (auto& a : m->allocs)
    if (a.base) cudaFree(a.base);
  if (m->scratch) cudaFree(m->scratch);
  if (m->timeline) cudaFree(m->timeline);
  for (cudaEvent_t e : m->ev)
    if (e) cudaEventDestroy(e);
  if (m->graph_exec) cudaGraphExecDestroy(m->graph_exec);
  if (m->graph) cudaGraphDestroy(m->graph);
  if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
  if (m->step_dev) cudaFree(m->step_dev);
  if (m->step_host) cudaFreeHost(m->step_host);
  delete m;
}

static msk_status check_bf16(const msk_bf16_desc& x, int64_t rows, int64_t cols) {
  if (x.data == nullptr) return MSK_ERR_INVALID_ARG;
  if (x.rows != rows || x.cols != cols) return MSK_ERR_SHAPE;
  const int64_t ld = x.ld_elems ? x.ld_elems : cols;
  if (ld < cols || ld % 8) return MSK_ERR_ALIGNMENT;
  if (!aligned16(x.data)) return MSK_ERR_ALIGNMENT;
  return MSK_OK;
}

extern "C" msk_status msk_load_layer(msk_model* m, int32_t layer, const msk_layer_weights* w, void* stream) {
  if (m == nullptr || w == nullptr) return MSK_ERR_INVALID_ARG;
  if (layer < 0 || layer >= m->dm.n_layers) return MSK_ERR_INVALID_ARG;
  const Dims& d = m->dm;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int qkv_rows = (d.Hq + 2 * d.Hkv) * d.hd;
  msk_status r;
  if ((r = check_bf16(w->attn_norm, 1, d.D)) != MSK_OK) return r;
  if ((r = check_bf16(w->moe_norm, 1, d.D)) != MSK_OK) return r;
  if ((r = check_bf16(w->w_qkv, qkv_rows, d.D)) != MSK_OK) return r;
  if ((r = check_bf16(w->w_o, d.D, (int64_t)d.Hq * d.hd)) != MSK_OK) return r;
  if ((r = check_bf16(w->w_pool, d.P, d.D)) != MSK_OK) return r;
  if ((r = check_bf16(w->w_router, d.E, d.P)) != MSK_OK) return r;
  if ((r = check_bf16(w->w_unpool, d.D, d.P)) != MSK_OK) return r;
  if (w->router_bias == nullptr || w->w_gate == nullptr || w->w_up == nullptr || w->w_down == nullptr)
    return MSK_ERR_INVALID_ARG;
  std::vector<const uint8_t*> srcs(3 * 2 * d.E);
  std::vector<float> ts(3 * d.E);
  for (int e = 0; e < d.E; ++e) {
    const msk_nvfp4_desc* ds[3] = {&w->w_gate[e], &w->w_up[e], &w->w_down[e]};
    const int64_t rows[3] = {d.I, d.I, d.P}, cols[3] = {d.P, d.P, d.I};
    for (int k = 0; k < 3; ++k) {
      if (ds[k]->packed == nullptr || ds[k]->scales == nullptr) return MSK_ERR_INVALID_ARG;
      if (ds[k]->rows != rows[k] || ds[k]->cols != cols[k]) return MSK_ERR_SHAPE;
      if (!aligned16(ds[k]->packed) || !aligned16(ds[k]->scales)) return MSK_ERR_ALIGNMENT;
      srcs[(e * 3 + k) * 2] = ds[k]->packed;
      srcs[(e * 3 + k) * 2 + 1] = ds[k]->scales;
      ts[e * 3 + k] = ds[k]->tensor_scale;
    }
  }
  // layout of this layer's allocation
  const size_t b_qkv = align_up(dense_tiled_bytes(qkv_rows, d.D), 256);
  const size_t b_o = align_up(dense_tiled_bytes(d.D, (int64_t)d.Hq * d.hd), 256);
  const size_t b_pool = align_up(dense_tiled_bytes(d.P, d.D), 256);
  const size_t b_r = align_up(dense_tiled_bytes(d.E, d.P), 256);
  const size_t b_un = align_up(dense_tiled_bytes(d.D, d.P), 256);
  const size_t b_norm = align_up((size_t)d.D * 2, 256);
  const size_t b_bias = align_up((size_t)d.E * 4, 256);
  const size_t b_ts = align_up((size_t)d.E * 3 * 4, 256);
  const size_t b_ex = (size_t)d.E * xexpert_bytes(d.P, d.I);
  const size_t total = b_qkv + b_o + b_pool + b_r + b_un + 2 * b_norm + b_bias + b_ts + b_ex;
  LayerAlloc& al = m->allocs[layer];
  if (al.base == nullptr) {
    if (cudaMalloc(&al.base, total) != cudaSuccess) {
      al.base = nullptr;
      return MSK_ERR_OOM;
    }
    al.bytes = total;
    m->weight_bytes += total;
  }
  uint8_t* p = static_cast<uint8_t*>(al.base);
  LayerDev& L = m->layers[layer];
  L.loaded = 0;
  L.w_qkv = p; p += b_qkv;
  L.w_o = p; p += b_o;
  L.w_pool = p; p += b_pool;
  L.w_router = p; p += b_r;
  L.w_unpool = p; p += b_un;
  L.attn_norm = reinterpret_cast<const uint16_t*>(p); p += b_norm;
  L.moe_norm = reinterpret_cast<const uint16_t*>(p); p += b_norm;
  L.router_bias = reinterpret_cast<const float*>(p); p += b_bias;
  L.ts = reinterpret_cast<const float*>(p); p += b_ts;
  L.experts = p;

  auto ld = [](const msk_bf16_desc& x) { return x.ld_elems ? x.ld_elems : x.cols; };
  MSK_CUDA(repack_dense(w->w_qkv.data, ld(w->w_qkv), qkv_rows, d.D, (void*)L.w_qkv, (d.Hq + d.Hkv) * d.hd, d.hd, st));
  MSK_CUDA(repack_dense(w->w_o.data, ld(w->w_o), d.D, d.Hq * d.hd, (void*)L.w_o, 0, d.hd, st));
  MSK_CUDA(repack_dense(w->w_pool.data, ld(w->w_pool), d.P, d.D, (void*)L.w_pool, 0, d.hd, st));
  MSK_CUDA(repack_dense(w->w_router.data, ld(w->w_router), d.E, d.P, (void*)L.w_router, 0, d.hd, st));
  MSK_CUDA(repack_dense(w->w_unpool.data, ld(w->w_unpool), d.D, d.P, (void*)L.w_unpool, 0, d.hd, st));
  MSK_CUDA(cudaMemcpyAsync((void*)L.attn_norm, w->attn_norm.data, (size_t)d.D * 2, cudaMemcpyDeviceToDevice, st));
  MSK_CUDA(cudaMemcpyAsync((void*)L.moe_norm, w->moe_norm.data, (size_t)d.D * 2, cudaMemcpyDeviceToDevice, st));
  MSK_CUDA(cudaMemcpyAsync((void*)L.router_bias, w->router_bias, (size_t)d.E * 4, cudaMemcpyDeviceToDevice, st));
  MSK_CUDA(cudaMemcpyAsync((void*)L.ts, ts.data(), ts.size() * 4, cudaMemcpyHostToDevice, st));
  void* tmp = nullptr;
  const size_t tmp_bytes = srcs.size() * sizeof(void*) + 16;
  if (cudaMalloc(&tmp, tmp_bytes) != cudaSuccess) return MSK_ERR_OOM;
  int* bad = reinterpret_cast<int*>(static_cast<uint8_t*>(tmp) + srcs.size() * sizeof(void*));
  msk_status rs = MSK_OK;
  int hbad = 0;
  if (cudaMemcpyAsync(tmp, srcs.data(), srcs.size() * sizeof(void*), cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemsetAsync(bad, 0, sizeof(int), st) != cudaSuccess ||
      repack_experts(tmp, d.E, d.P, d.I, (void*)L.experts, bad, st) != cudaSuccess ||
      cudaMemcpyAsync(&hbad, bad, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    rs = MSK_ERR_CUDA;
  cudaFree(tmp);
  if (rs != MSK_OK) return rs;
  if (hbad) return MSK_ERR_BAD_SCALE;
  L.loaded = 1;
  return MSK_OK;
}

static msk_status check_positions(const msk_model* m, const int32_t* positions) {
  if (positions == nullptr) return MSK_ERR_INVALID_ARG;
  const Dims& d = m->dm;
  for (int t = 0; t < d.T; ++t)
    if (positions[t] != positions[0] + t) return MSK_ERR_INVALID_ARG;
  if (positions[0] < 0 || positions[0] + d.T > d.max_seq) return MSK_ERR_INVALID_ARG;
  return MSK_OK;
}

static void fill_args(msk_model* m, LaunchArgs& a, int layer, void* hidden, void* kv, int pos0, int prologue,
                      const int32_t* prev, int32_t* rout, const int32_t* parents) {
  const Dims& d = m->dm;
  a.dm = d;
  a.cur = m->layers[layer];
  tree_masks(parents, d.T, a.cur.window, a.depth, a.vis);  // (parents validated by the caller)
  a.has_next = layer + 1 < d.n_layers;
  a.nxt = a.has_next ? m->layers[layer + 1] : m->layers[layer];
  a.s = m->s;
  a.hidden = static_cast<uint16_t*>(hidden);
  const size_t layer_elems = (size_t)2 * d.Hkv * d.max_seq * d.hd;
  a.kv_cur = static_cast<uint16_t*>(kv) + (size_t)layer * layer_elems;
  a.kv_nxt = a.has_next ? a.kv_cur + layer_elems : nullptr;
  a.kv_nxt_ro = a.kv_nxt;
  a.pos0 = pos0;
  a.prologue = prologue;
  a.prev_routing = prev;
  a.routing_out = rout;
  a.budget_ns = m->budget;
  a.timeline = m->timing && m->timeline ? m->timeline + (size_t)layer * d.nctas * kTimelineSlots : nullptr;
  a.inject_bar = m->inject_bar;
  a.inject_cta = m->inject_cta;
  a.kv_prefetch_rows = m->kv_prefetch_rows;
  a.step = nullptr;
  a.kv_z0 = layer * 2 * d.Hkv;
  a.kv_map = m->kv_map;  // (prepared for this cache by the caller)
}

static msk_status finish(msk_model* m, cudaStream_t st) {
  const cudaError_t se = cudaStreamSynchronize(st);
  if (se != cudaSuccess) {
    if (getenv("MSK_VERBOSE_ERRORS") != nullptr) fprintf(stderr, "msk: %s\n", cudaGetErrorString(se));
    return MSK_ERR_CUDA;
  }
  uint32_t err[4] = {0, 0, 0, 0};
  if (cudaMemcpy(err, m->s.err, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) return MSK_ERR_CUDA;
  if (err[0] != 0) {
    if (getenv("MSK_VERBOSE_ERRORS") != nullptr)
      fprintf(stderr, "msk: device error code %u in phase %d (block %u)\n", err[0], (int)err[1], err[2]);
    // reset the device synchronisation state for the next call
    cudaMemset(m->s.bar, 0, 64);
    cudaMemset(m->s.err, 0, 64);
    cudaMemset(m->s.x1_done, 0, (size_t)(2 * m->dm.E + 2) * 4);
    cudaDeviceSynchronize();
    return MSK_ERR_TIMEOUT;
  }
  return MSK_OK;
}

// Validates a candidate tree (parents[t] in [-1, t)) and the cached length.
static msk_status check_tree(const msk_model* m, int32_t cache_len, const int32_t* parents) {
  if (parents == nullptr) return MSK_ERR_INVALID_ARG;
  const Dims& d = m->dm;
  for (int t = 0; t < d.T; ++t)
    if (parents[t] < -1 || parents[t] >= t) return MSK_ERR_INVALID_ARG;
  if (cache_len < 0 || cache_len + d.T > d.max_seq) return MSK_ERR_INVALID_ARG;
  return MSK_OK;
}

// One launch; parents == nullptr is the chain.
static msk_status layer_step_impl(msk_model* m, int32_t layer, void* hidden, void* kv_cache, int32_t pos0,
                                  const int32_t* parents, const int32_t* prev_routing, int32_t* routing_out,
                                  int32_t run_prologue, void* stream) {
  if (!aligned16(hidden) || !aligned16(kv_cache)) return MSK_ERR_ALIGNMENT;
  if (!m->layers[layer].loaded) return MSK_ERR_NOT_LOADED;
  if (layer + 1 < m->dm.n_layers && !m->layers[layer + 1].loaded) return MSK_ERR_NOT_LOADED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!prepare_kv_map(m, kv_cache)) return MSK_ERR_CUDA;
  LaunchArgs a;
  fill_args(m, a, layer, hidden, kv_cache, pos0, run_prologue ? 1 : 0, prev_routing, routing_out, parents);
  if (m->launch_timing) cudaEventRecord(m->ev[0], st);
  if (launch_layer(a, m->timing, false, st) != cudaSuccess) return MSK_ERR_CUDA;
  if (m->launch_timing) cudaEventRecord(m->ev[1], st);
  m->last_launches = 1;
  m->last_first = layer;
  return finish(m, st);
}

// The whole step; parents == nullptr is the chain.
static msk_status decode_step_impl(msk_model* m, void* hidden, void* kv_cache, int32_t pos0, const int32_t* parents,
                                   const int32_t* prev_routing, int32_t* routing_out, void* stream) {
  if (!aligned16(hidden) || !aligned16(kv_cache)) return MSK_ERR_ALIGNMENT;
  const Dims& d = m->dm;
  for (int l = 0; l < d.n_layers; ++l)
    if (!m->layers[l].loaded) return MSK_ERR_NOT_LOADED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!prepare_kv_map(m, kv_cache)) return MSK_ERR_CUDA;
  const size_t rk = (size_t)d.T * d.topk;
  for (int l = 0; l < d.n_layers; ++l) {
    LaunchArgs a;
    fill_args(m, a, l, hidden, kv_cache, pos0, l == 0 ? 1 : 0, prev_routing ? prev_routing + l * rk : nullptr,
              routing_out ? routing_out + l * rk : nullptr, parents);
    if (m->launch_timing) cudaEventRecord(m->ev[2 * l], st);
    // (with per-launch events between them the launches are not chained)
    const cudaError_t le = launch_layer(a, m->timing, l > 0 && !m->launch_timing, st);
    if (le != cudaSuccess) {
      if (getenv("MSK_VERBOSE_ERRORS") != nullptr)
        fprintf(stderr, "msk: launch of layer %d: %s\n", l, cudaGetErrorString(le));
      return MSK_ERR_CUDA;
    }
    if (m->launch_timing) cudaEventRecord(m->ev[2 * l + 1], st);
  }
  m->last_launches = d.n_layers;
  m->last_first = 0;
  return finish(m, st);
}

extern "C" msk_status msk_layer_step(msk_model* m, int32_t layer, void* hidden, void* kv_cache, const int32_t* positions,
                                     const int32_t* prev_routing, int32_t* routing_out, int32_t run_prologue,
                                     void* stream) {
  if (m == nullptr || hidden == nullptr || kv_cache == nullptr) return MSK_ERR_INVALID_ARG;
  if (layer < 0 || layer >= m->dm.n_layers) return MSK_ERR_INVALID_ARG;
  msk_status r = check_positions(m, positions);
  if (r != MSK_OK) return r;
  return layer_step_impl(m, layer, hidden, kv_cache, positions[0], nullptr, prev_routing, routing_out, run_prologue,
                         stream);
}

extern "C" msk_status msk_decode_step(msk_model* m, void* hidden, void* kv_cache, const int32_t* positions,
                                      const int32_t* prev_routing, int32_t* routing_out, void* stream) {
  if (m == nullptr || hidden == nullptr || kv_cache == nullptr) return MSK_ERR_INVALID_ARG;
  msk_status r = check_positions(m, positions);
  if (r != MSK_OK) return r;
  return decode_step_impl(m, hidden, kv_cache, positions[0], nullptr, prev_routing, routing_out, stream);
}

extern "C" msk_status msk_layer_step_tree(msk_model* m, int32_t layer, void* hidden, void* kv_cache,
                                          int32_t cache_len, const int32_t* parents, const int32_t* prev_routing,
                                          int32_t* routing_out, int32_t run_prologue, void* stream) {
  if (m == nullptr || hidden == nullptr || kv_cache == nullptr) return MSK_ERR_INVALID_ARG;
  if (layer < 0 || layer >= m->dm.n_layers) return MSK_ERR_INVALID_ARG;
  msk_status r = check_tree(m, cache_len, parents);
  if (r != MSK_OK) return r;
  return layer_step_impl(m, layer, hidden, kv_cache, cache_len, parents, prev_routing, routing_out, run_prologue,
                         stream);
}

extern "C" msk_status msk_decode_step_tree(msk_model* m, void* hidden, void* kv_cache, int32_t cache_len,
                                           const int32_t* parents, const int32_t* prev_routing, int32_t* routing_out,
                                           void* stream) {
  if (m == nullptr || hidden == nullptr || kv_cache == nullptr) return MSK_ERR_INVALID_ARG;
  msk_status r = check_tree(m, cache_len, parents);
  if (r != MSK_OK) return r;
  return decode_step_impl(m, hidden, kv_cache, cache_len, parents, prev_routing, routing_out, stream);
}

extern "C" msk_status msk_step_graph_capture(msk_model* m, void* hidden, void* kv_cache,
                                             const int32_t* prev_routing, int32_t* routing_out) {
  if (m == nullptr || hidden == nullptr || kv_cache == nullptr) return MSK_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(kv_cache)) return MSK_ERR_ALIGNMENT;
  const Dims& d = m->dm;
  for (int l = 0; l < d.n_layers; ++l)
    if (!m->layers[l].loaded) return MSK_ERR_NOT_LOADED;
  if (m->step_dev == nullptr && cudaMalloc(&m->step_dev, sizeof(StepInfo)) != cudaSuccess) {
    m->step_dev = nullptr;
    return MSK_ERR_OOM;
  }
  if (m->step_host == nullptr && cudaMallocHost(&m->step_host, sizeof(StepInfo)) != cudaSuccess) {
    m->step_host = nullptr;
    return MSK_ERR_OOM;
  }
  if (m->cap_stream == nullptr) MSK_CUDA(cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking));
  MSK_CUDA(prepare_launch());  // kernel attributes are set outside the capture
  if (!prepare_kv_map(m, kv_cache)) return MSK_ERR_CUDA;
  if (m->graph_exec) {
    cudaGraphExecDestroy(m->graph_exec);
    m->graph_exec = nullptr;
  }
  if (m->graph) {
    cudaGraphDestroy(m->graph);
    m->graph = nullptr;
  }
  MSK_CUDA(cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
  const size_t rk = (size_t)d.T * d.topk;
  bool ok = true;
  for (int l = 0; l < d.n_layers && ok; ++l) {
    LaunchArgs a;
    fill_args(m, a, l, hidden, kv_cache, 0, l == 0 ? 1 : 0, prev_routing ? prev_routing + l * rk : nullptr,
              routing_out ? routing_out + l * rk : nullptr, nullptr);
    a.step = m->step_dev;
    a.timeline = nullptr;
    ok = launch_layer(a, false, l > 0, m->cap_stream) == cudaSuccess;
  }
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(m->cap_stream, &g);
  if (!ok || ec != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return MSK_ERR_CUDA;
  }
  if (cudaGraphInstantiate(&m->graph_exec, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    m->graph_exec = nullptr;
    return MSK_ERR_CUDA;
  }
  m->graph = g;
  return MSK_OK;
}

extern "C" msk_status msk_step_graph_launch(msk_model* m, int32_t cache_len, const int32_t* parents, void* stream) {
  if (m == nullptr) return MSK_ERR_INVALID_ARG;
  if (m->graph_exec == nullptr) return MSK_ERR_NOT_LOADED;
  const Dims& d = m->dm;
  if (parents != nullptr) {
    const msk_status r = check_tree(m, cache_len, parents);
    if (r != MSK_OK) return r;
  } else if (cache_len < 0 || cache_len + d.T > d.max_seq) {
    return MSK_ERR_INVALID_ARG;
  }
  StepInfo* h = m->step_host;
  h->pos0 = cache_len;
  tree_masks(parents, d.T, 0, h->depth, h->vis[0]);
  tree_masks(parents, d.T, m->cfg.window, h->depth, h->vis[1]);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MSK_CUDA(cudaMemcpyAsync(m->step_dev, h, sizeof(StepInfo), cudaMemcpyHostToDevice, st));
  MSK_CUDA(cudaGraphLaunch(m->graph_exec, st));
  m->last_launches = d.n_layers;
  m->last_first = 0;
  return finish(m, st);
}

extern "C" msk_status msk_set_timing(msk_model* m, int32_t enable) {
  if (m == nullptr) return MSK_ERR_INVALID_ARG;
  if (enable && m->timeline == nullptr) {
    const size_t n = (size_t)m->dm.n_layers * m->dm.nctas * kTimelineSlots;
    if (cudaMalloc(&m->timeline, n * 8) != cudaSuccess) {
      m->timeline = nullptr;
      return MSK_ERR_OOM;
    }
    cudaMemset(m->timeline, 0, n * 8);
  }
  m->timing = enable != 0;
  return MSK_OK;
}

extern "C" msk_status msk_get_timeline(msk_model* m, uint64_t* host_out, size_t cap, size_t* n, int32_t* n_launches,
                                       int32_t* n_ctas) {
  if (m == nullptr || n == nullptr) return MSK_ERR_INVALID_ARG;
  *n = 0;
  if (n_ctas) *n_ctas = m->dm.nctas;
  if (n_launches) *n_launches = m->last_launches;
  if (m->timeline == nullptr) return MSK_OK;
  const size_t want = (size_t)m->last_launches * m->dm.nctas * kTimelineSlots;
  const size_t k = std::min(want, cap);
  if (k && host_out) {
    const unsigned long long* src = m->timeline + (size_t)m->last_first * m->dm.nctas * kTimelineSlots;
    if (cudaMemcpy(host_out, src, k * 8, cudaMemcpyDeviceToHost) != cudaSuccess) return MSK_ERR_CUDA;
  }
  *n = k;
  return MSK_OK;
}

extern "C" msk_status msk_set_launch_timing(msk_model* m, int32_t enable) {
  if (m == nullptr) return MSK_ERR_INVALID_ARG;
  if (enable && m->ev.empty()) {
    m->ev.assign(2 * (size_t)m->dm.n_layers, nullptr);
    for (auto& e : m->ev)
      if (cudaEventCreate(&e) != cudaSuccess) return MSK_ERR_CUDA;
  }
  m->launch_timing = enable != 0;
  return MSK_OK;
}

extern "C" msk_status msk_get_launch_ms(msk_model* m, float* host_out, int32_t cap, int32_t* n) {
  if (m == nullptr || n == nullptr) return MSK_ERR_INVALID_ARG;
  *n = 0;
  if (m->ev.empty() || host_out == nullptr) return MSK_OK;
  const int k = std::min(cap, m->last_launches);
  for (int i = 0; i < k; ++i) {
    if (cudaEventSynchronize(m->ev[2 * i + 1]) != cudaSuccess) return MSK_ERR_CUDA;
    if (cudaEventElapsedTime(&host_out[i], m->ev[2 * i], m->ev[2 * i + 1]) != cudaSuccess) return MSK_ERR_CUDA;
  }
  *n = k;
  return MSK_OK;
}

extern "C" msk_status msk_set_wait_budget(msk_model* m, uint64_t ns) {
  if (m == nullptr) return MSK_ERR_INVALID_ARG;
  m->budget = ns ? ns : kDefaultBudgetNs;
  return MSK_OK;
}

extern "C" msk_status msk_set_fault_injection(msk_model* m, int32_t barrier, int32_t cta) {
  if (m == nullptr) return MSK_ERR_INVALID_ARG;
  m->inject_bar = barrier;
  m->inject_cta = cta;
  return MSK_OK;
}

extern "C" msk_status msk_debug_scratch(msk_model* m, int32_t which, void* dst, size_t bytes, size_t* copied,
                                        void* stream) {
  if (m == nullptr || dst == nullptr || copied == nullptr) return MSK_ERR_INVALID_ARG;
  const Dims& d = m->dm;
  const size_t tk = (size_t)d.T * d.topk;
  const void* src = nullptr;
  size_t n = 0;
  switch (which) {
    case 0: src = m->s.q_stash; n = (size_t)d.T * d.Hq * d.hd * 2; break;
    case 1: src = m->s.attn_o; n = (size_t)d.T * d.Hq * d.hd * 2; break;
    case 2: src = m->s.h1; n = (size_t)d.T * d.D * 2; break;
    case 3: src = m->s.pooled; n = (size_t)d.T * d.P * 2; break;
    case 4: src = m->s.logits; n = (size_t)d.T * d.E * 4; break;
    case 5: src = m->s.sq_codes; n = tk * (d.I / 2); break;
    case 6: src = m->s.sq_scales; n = tk * (d.I / 16); break;
    case 7: src = m->s.y; n = tk * d.P * 2; break;
    case 8: src = m->s.mvec; n = (size_t)d.T * d.P * 2; break;
    case 9: src = m->s.pf_out; n = 33 * 4; break;
    default: return MSK_ERR_INVALID_ARG;
  }
  n = std::min(n, bytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MSK_CUDA(cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToDevice, st));
  MSK_CUDA(cudaStreamSynchronize(st));
  *copied = n;
  return MSK_OK;
}

extern "C" msk_status msk_debug_dequant(msk_model* m, int32_t layer, int32_t expert, int32_t which, float* out,
                                        void* stream) {
  if (m == nullptr || out == nullptr || layer < 0 || layer >= m->dm.n_layers) return MSK_ERR_INVALID_ARG;
  if (expert < 0 || expert >= m->dm.E || which < 0 || which > 2) return MSK_ERR_INVALID_ARG;
  if (!m->layers[layer].loaded) return MSK_ERR_NOT_LOADED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MSK_CUDA(debug_dequant(m->layers[layer].experts, m->layers[layer].ts, m->dm.P, m->dm.I, expert, which, out, st));
  MSK_CUDA(cudaStreamSynchronize(st));
  return MSK_OK;
}

extern "C" msk_status msk_debug_convert(const float* x, int64_t n, uint8_t* e2m1, uint8_t* e4m3, void* stream) {
  if (x == nullptr || e2m1 == nullptr || e4m3 == nullptr || n < 0) return MSK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (n > 0) MSK_CUDA(debug_convert(x, n, e2m1, e4m3, st));
  MSK_CUDA(cudaStreamSynchronize(st));
  return MSK_OK;
}

extern "C" msk_status msk_debug_quantize(const float* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* scales,
                                         void* stream) {
  if (x == nullptr || codes == nullptr || scales == nullptr || rows <= 0 || cols <= 0 || cols % 16)
    return MSK_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MSK_CUDA(debug_quantize(x, rows, cols, codes, scales, st));
  MSK_CUDA(cudaStreamSynchronize(st));
  return MSK_OK;
}

extern "C" msk_status msk_debug_fp4_gemm(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* b_codes,
                                         const uint8_t* b_scales, int32_t b_rows, int32_t K, float* d, void* stream) {
  if (a_codes == nullptr || a_scales == nullptr || b_codes == nullptr || b_scales == nullptr || d == nullptr)
    return MSK_ERR_INVALID_ARG;
  if (K < 128 || K > 2048 || K % 128 || b_rows < 1 || b_rows > kUN) return MSK_ERR_SHAPE;
  if (!aligned16(a_codes) || !aligned16(b_codes)) return MSK_ERR_ALIGNMENT;
  int dev = 0;
  MSK_CUDA(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  MSK_CUDA(cudaGetDeviceProperties(&prop, dev));
  if (!(prop.major == 10 && prop.minor == 3)) return MSK_ERR_UNSUPPORTED_DEVICE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* err = nullptr;
  if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) return MSK_ERR_OOM;
  uint32_t herr = 0;
  msk_status r = MSK_OK;
  if (cudaMemsetAsync(err, 0, sizeof(uint32_t), st) != cudaSuccess ||
      debug_fp4_tile(a_codes, a_scales, b_codes, b_scales, b_rows, K, d, err, st) != cudaSuccess ||
      cudaMemcpyAsync(&herr, err, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    r = MSK_ERR_CUDA;
  cudaFree(err);
  if (r == MSK_OK && herr) r = MSK_ERR_TIMEOUT;
  return r;
}

extern "C" msk_status msk_get_info(msk_model* m, int32_t* n_ctas, int64_t* device_bytes) {
  if (m == nullptr) return MSK_ERR_INVALID_ARG;
  if (n_ctas) *n_ctas = m->dm.nctas;
  if (device_bytes) *device_bytes = (int64_t)(m->scratch_bytes + m->weight_bytes);
  return MSK_OK;
}
