// The persistent layer kernel: one launch = attention(l) .. MoE(l) ..
// QKV(l+1) + KV write ([orcarouter] "Dove si colloca il confine del
// kernel"; [newruntime] "What happened").  One block per SM, 9 warps with
// fixed roles: warp 8 streams weights (producer), warps 0..7 compute.
// Phases are separated by a bounded grid barrier; the producer does not wait
// on it and keeps the weight stream going across phase boundaries.
#include <cuda_runtime.h>

#include "msk_phases_moe.cuh"

namespace msk {

template <int HD, bool TIMING>
__global__ void __launch_bounds__(kThreads, 1) msk_layer_kernel(const __grid_constant__ LaunchArgs args) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctx c;
  c.a = &args;
  c.smem = smem;
  c.misc = reinterpret_cast<Misc*>(smem + kOffMisc);
  c.sbase = smem_u32(smem);
  c.cta = blockIdx.x;
  c.nctas = gridDim.x;
  c.tid = threadIdx.x;
  c.warp = threadIdx.x >> 5;
  c.lane = threadIdx.x & 31;
  c.seq = 0;
  c.nbar = 0;
  const LaunchArgs& a = args;
  const Dims& d = a.dm;
  if (c.tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(c.bar(BAR_FULL + i), 1);
      mbar_init(c.bar(BAR_EMPTY + i), kConsWarps);
    }
    mbar_init(c.bar(BAR_KV), 1);
    mbar_init(c.bar(BAR_KV + 1), 1);
    mbar_init(c.bar(BAR_DISPATCH), 1);
    c.misc->abort = 0;
    c.misc->n_used = 0;
    c.misc->zero = 0;
    c.misc->spare = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (c.warp == kConsWarps) {
    producer(c);
    return;
  }
  auto mark = [&](int slot) {
    if constexpr (TIMING) stamp(c, slot);
  };
  mark(PH_START);
  const int qkv_rows = (d.Hq + 2 * d.Hkv) * d.hd;
  if (a.prologue || a.has_next) rope_table(c);
  if (a.prologue) {
    if (!grid_barrier(c, PH_PRO_QKV)) return;
    mark(PH_PRO_QKV);
    stage_rmsnorm(c, a.hidden, a.cur.attn_norm, d.D);
    named_bar(1, kConsThreads);
    EpiQKV epi{a.s.rope, a.s.q_stash, a.kv_cur, d.T, d.Hq, d.Hkv, d.hd, d.max_seq, a.pos0};
    dense_phase(c, a.cur.w_qkv, qkv_rows, d.D, epi);
    if (!grid_barrier(c, PH_PRO_QKV)) return;
  }
  mark(PH_ATTN);
  attention_phase<HD>(c);
  if (!grid_barrier(c, PH_ATTN)) return;
  mark(PH_COMBINE);
  combine_phase<HD>(c);
  if (!grid_barrier(c, PH_COMBINE)) return;
  mark(PH_OPROJ);
  {
    stage_copy(c, a.s.attn_o, d.Hq * d.hd);
    named_bar(1, kConsThreads);
    EpiResidual epi{a.hidden, a.s.h1, d.T, d.D};
    dense_phase(c, a.cur.w_o, d.D, d.Hq * d.hd, epi);
  }
  if (!grid_barrier(c, PH_OPROJ)) return;
  mark(PH_POOL);
  {
    stage_rmsnorm(c, a.s.h1, a.cur.moe_norm, d.D);
    named_bar(1, kConsThreads);
    EpiStore epi{a.s.pooled, d.T, d.P};
    dense_phase(c, a.cur.w_pool, d.P, d.D, epi);
  }
  if (!grid_barrier(c, PH_POOL)) return;
  mark(PH_ROUTER);
  {
    stage_copy(c, a.s.pooled, d.P);
    named_bar(1, kConsThreads);
    EpiRouter epi{a.s.logits, a.cur.router_bias, d.T, d.E};
    dense_phase(c, a.cur.w_router, d.E, d.P, epi);
  }
  if (!grid_barrier(c, PH_ROUTER)) return;
  mark(PH_TOPK);
  topk_dispatch(c);
  mark(PH_GEMM1);
  gemm1_phase(c);
  if (!grid_barrier(c, PH_GEMM1)) return;
  mark(PH_GEMM2);
  gemm2_phase(c);
  if (!grid_barrier(c, PH_GEMM2)) return;
  mark(PH_MCOMB);
  mcomb_phase(c);
  if (!grid_barrier(c, PH_MCOMB)) return;
  mark(PH_UNPOOL);
  {
    stage_copy(c, a.s.mvec, d.P);
    named_bar(1, kConsThreads);
    EpiResidual epi{a.s.h1, a.hidden, d.T, d.D};
    dense_phase(c, a.cur.w_unpool, d.D, d.P, epi);
  }
  if (a.has_next) {
    if (!grid_barrier(c, PH_UNPOOL)) return;
    mark(PH_QKV);
    stage_rmsnorm(c, a.hidden, a.nxt.attn_norm, d.D);
    named_bar(1, kConsThreads);
    EpiQKV epi{a.s.rope, a.s.q_stash, a.kv_nxt, d.T, d.Hq, d.Hkv, d.hd, d.max_seq, a.pos0};
    dense_phase(c, a.nxt.w_qkv, qkv_rows, d.D, epi);
  }
  named_bar(1, kConsThreads);
  mark(PH_END);
}

template <int HD, bool TIMING>
static cudaError_t launch_t(const LaunchArgs& args, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(msk_layer_kernel<HD, TIMING>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(args.dm.nctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, msk_layer_kernel<HD, TIMING>, args);
}

cudaError_t launch_layer(const LaunchArgs& args, bool timing, cudaStream_t st) {
  if (args.dm.hd == 128) return timing ? launch_t<128, true>(args, st) : launch_t<128, false>(args, st);
  return timing ? launch_t<64, true>(args, st) : launch_t<64, false>(args, st);
}

int smem_bytes() { return kSmemBytes; }

}  // namespace msk
