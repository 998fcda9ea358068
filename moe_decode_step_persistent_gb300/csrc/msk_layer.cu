// The persistent layer kernel: one launch = attention(l) .. MoE(l) ..
// QKV(l+1) + KV write ([orcarouter] "Dove si colloca il confine del
// kernel"; [newruntime] "What happened").  One block per SM, 11 warps with
// fixed roles: warp 8 streams weights (producer), warps 9 and 10 issue the
// expert GEMMs' tensor-core operations (one lane each, half of every weight
// stage's MMAs each: one issuing thread's instruction latency, not the
// tensor core, bounds the issue rate), warps 0..7 compute.
// Phases are separated by a bounded grid barrier; the producer does not wait
// on it and keeps the weight stream going across phase boundaries.  The
// expert GEMMs run on the fifth-generation tensor cores with their
// accumulators in tensor memory (allocated for the launch by warp 0).
#include <cuda_runtime.h>

#include "msk_phases_moe.cuh"

namespace msk {

// The compute warps' phases of one launch; returns early (uniformly over the
// compute warps) when a grid barrier reports an abort.
template <int HD, bool TIMING>
__device__ __forceinline__ void layer_phases(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  auto mark = [&](int slot) {
    if constexpr (TIMING) stamp(c, slot);
  };
  // slot 16 + phase: the block finished the phase's work (before the barrier)
  auto done = [&](int phase) {
    if constexpr (TIMING) {
      named_bar(1, kConsThreads);
      stamp(c, 16 + phase);
    }
  };
  mark(PH_START);
  if (aborted(c)) return;  // (uniform: set before the block-wide barrier at launch start)
  // the top-k's expert -> token masks (set there by shared-memory atomics)
  for (int e = c.tid(); e < 256; e += kConsThreads) c.misc()->tok_mask[e] = 0u;
  const int qkv_rows = (d.Hq + 2 * d.Hkv) * d.hd;
  // the step's RoPE table (every launch of a step has the same positions):
  // computed by the launch that runs the prologue, reused by the later ones
  if (a.prologue) rope_table(c);
  if (a.prologue) {
    done(PH_PRO_QKV);
    if (!grid_barrier(c, PH_PRO_QKV)) return;
    mark(PH_PRO_QKV);
    stage_rmsnorm(c, a.hidden, a.cur.attn_norm, d.D, false);
    named_bar(1, kConsThreads);
    dense_phase(c, a.cur.w_qkv, qkv_rows, d.D, OP_QKV_CUR);
    done(PH_PRO_QKV);
    if (!grid_barrier(c, PH_PRO_QKV)) return;
  }
  mark(PH_ATTN);
  attention_phase<HD>(c);
  done(PH_ATTN);
  if (!grid_barrier(c, PH_ATTN)) return;
  mark(PH_COMBINE);
  combine_phase<HD>(c);
  done(PH_COMBINE);
  if (!grid_barrier(c, PH_COMBINE)) return;
  mark(PH_OPROJ);
  stage_issue(c, a.s.attn_o, d.Hq * d.hd);
  named_bar(1, kConsThreads);
  dense_phase(c, a.cur.w_o, d.D, d.Hq * d.hd, OP_OPROJ);
  done(PH_OPROJ);
  if (!grid_barrier(c, PH_OPROJ)) return;
  mark(PH_POOL);
  stage_rmsnorm(c, a.s.h1, a.cur.moe_norm, d.D, true);
  named_bar(1, kConsThreads);
  dense_phase(c, a.cur.w_pool, d.P, d.D, OP_POOL);
  done(PH_POOL);
  if (!grid_barrier(c, PH_POOL)) return;
  mark(PH_ROUTER);
  if (c.tid() == 0) mbar_arrive(c.bar(BAR_HOT));  // the producer's lanes may prefetch the hot experts
  stage_issue(c, a.s.pooled, d.P);
  named_bar(1, kConsThreads);
  dense_phase(c, a.cur.w_router, d.E, d.P, OP_ROUTER);
  quantize_pooled(c);
  done(PH_ROUTER);
  if (!grid_barrier(c, PH_ROUTER)) return;
  mark(PH_TOPK);
  topk_dispatch(c);
  // the routing is known (and the router phase consumed every ring tile):
  // the producer may stream the expert stages
  if (c.tid() == 0) mbar_arrive(c.bar(BAR_XGO));
  // both expert GEMMs, their units claimed from one queue (no grid barrier
  // between them: GEMM2's units are released as their experts' GEMM1 parts
  // complete)
  mark(PH_GEMM1);
  expert_gemms(c);
  done(PH_GEMM2);
  if (!grid_barrier(c, PH_GEMM2)) return;
  mark(PH_MCOMB);
  moe_combine_phase(c);
  done(PH_MCOMB);
  if (!grid_barrier(c, PH_MCOMB)) return;
  mark(PH_UNPOOL);
  stage_issue(c, a.s.mvec, d.P);
  named_bar(1, kConsThreads);
  dense_phase(c, a.cur.w_unpool, d.D, d.P, OP_UNPOOL);
  if (a.has_next) {
    done(PH_UNPOOL);
    if (!grid_barrier(c, PH_UNPOOL)) return;
    mark(PH_QKV);
    stage_rmsnorm(c, a.hidden, a.nxt.attn_norm, d.D, true);
    named_bar(1, kConsThreads);
    dense_phase(c, a.nxt.w_qkv, qkv_rows, d.D, OP_QKV_NXT);
  }
  done(a.has_next ? PH_QKV : PH_UNPOOL);
  named_bar(1, kConsThreads);
  mark(PH_END);
}

template <int HD, bool TIMING>
__global__ void __launch_bounds__(kThreads, 1) msk_layer_kernel(const __grid_constant__ LaunchArgs args) {
  // chained launches: this launch's blocks take the SMs as the previous
  // launch's blocks leave, and wait at grid_dep_wait until all of its work
  // is visible; the next launch may be queued right away (its blocks cannot
  // become resident before this launch's blocks exit).  The set-up that
  // reads nothing the previous launch writes runs before the wait: the
  // argument copy (the step record, when there is one, is written by a
  // host copy ahead of the step's first launch), the tensor-memory
  // allocation and the mbarriers.
  stage_args(args);
  Ctx c;
  if (c.warp() == 0) {
    // the expert GEMMs' accumulators and scale factors (one block per SM,
    // so the allocation never waits)
    tmem_alloc(smem_u32(&c.misc()->tmem), kTmemCols);
    tmem_relinquish();
  }
  if (c.tid() == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(c.bar(BAR_FULL + i), 1);
      mbar_init(c.bar(BAR_EMPTY + i), kConsWarps);
    }
    mbar_init(c.bar(BAR_XGO), 1);
    mbar_init(c.bar(BAR_HOT), 1);
    mbar_init(c.bar(BAR_STG), 1);
    for (int i = 0; i < kSegs; ++i) mbar_init(c.bar(BAR_SEG + i), 1);
    for (int i = 0; i < kAttnStages; ++i) mbar_init(c.bar(BAR_KV + i), 1);
    c.misc()->kvmap = reinterpret_cast<unsigned long long>(&args.kv_map);
    prefetch_tensormap(&args.kv_map);
    for (int i = 0; i < kXSlots; ++i) {
      mbar_init(c.bar(BAR_XFULL + i), 1);
      mbar_init(c.bar(BAR_XEMPTY + i), kMmaIssuers);
    }
    for (int i = 0; i < kAccs; ++i) {
      mbar_init(c.bar(BAR_ACCF + i), kMmaIssuers);
      mbar_init(c.bar(BAR_ACCE + i), kConsWarps);
    }
    mbar_init(c.bar(BAR_TCDONE), kMmaIssuers);
    for (int i = 0; i < 2; ++i) {
      mbar_init(c.bar(BAR_QFULL + i), 1);
      mbar_init(c.bar(BAR_QEMPTY + i), 1 + kMmaIssuers);
      mbar_init(c.bar(BAR_B2RDY + i), 1);
      mbar_init(c.bar(BAR_BFREE + i), kMmaIssuers);
    }
    mbar_fence_init();
  }
  if constexpr (TIMING) stamp(c, 29);
  grid_dep_wait();
  grid_dep_launch();
  if constexpr (TIMING) stamp(c, 16);
  c.seq = 0;
  c.nbar = 0;
  c.xseq = 0;
  c.xunit = 0;
  c.nstg = 0;
  c.sg = 0;
  c.bar0 = 0ull;
  if (c.tid() == 0) {
    // a launch that starts after an earlier launch of the call recorded an
    // error does nothing: the grid-barrier count may then have missed
    // arrivals (the host resets it once the call returns), and barriers
    // based on it would not hold the blocks together.  (The error word's
    // load is issued first, so that it is in flight with the acquiring load
    // of the barrier count.)
    const uint32_t err = ld_relaxed_gpu(args.s.err);
    c.bar0 = grid_barrier_base(args.s.bar);
    c.misc()->abort = err != 0u ? 1 : 0;
    c.misc()->n_used = 0;
    c.misc()->zero = 0;
    c.misc()->spare = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (c.warp() == kProducerWarp) {
    producer(c);
    return;
  }
  if (c.warp() >= kMmaWarp) {
    mma_warp(c, c.warp() - kMmaWarp);
    return;
  }
  layer_phases<HD, TIMING>(c);
  // release the tensor memory once every tcgen05 operation of the launch
  // has completed (each MMA warp's last commit tracks all of its own; the
  // barrier counts both; bounded; with the abort flag raised, an MMA warp
  // stops waiting and commits)
  if (c.tid() == 0) {
    *(volatile int*)&c.misc()->abort = 1;  // the launch is over: release a waiting MMA warp
    mbar_wait(c.bar(BAR_TCDONE), 0, gtimer() + 20000000ull, &c.misc()->zero);
  }
  tc_fence_before();
  named_bar(1, kConsThreads);
  tc_fence_after();
  if (c.warp() == 0) tmem_dealloc(c.misc()->tmem, kTmemCols);
}

template <int HD, bool TIMING>
static cudaError_t configure_t() {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(msk_layer_kernel<HD, TIMING>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return cudaSuccess;
}

template <int HD, bool TIMING>
static cudaError_t launch_t(const LaunchArgs& args, bool chained, cudaStream_t st) {
  cudaError_t e = configure_t<HD, TIMING>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(args.dm.nctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  // A step's first launch is cooperative (the grid barriers need every
  // block resident: one per SM).  A chained launch is a programmatic
  // dependent launch instead: a cooperative launch starts only once every SM
  // is free, while a dependent one places each block as the previous
  // launch's block on that SM exits; those blocks never wait on this launch,
  // so every block of it becomes resident.  (Were one not to, the grid
  // barrier's deadline would end the launch with an error.)
  cudaLaunchAttribute attr[1];
  if (chained) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, msk_layer_kernel<HD, TIMING>, args);
}

// chained: the launch follows another layer launch of the same step on the
// stream (programmatic dependent launch).
cudaError_t launch_layer(const LaunchArgs& args, bool timing, bool chained, cudaStream_t st) {
  if (args.dm.hd == 128) return timing ? launch_t<128, true>(args, chained, st) : launch_t<128, false>(args, chained, st);
  return timing ? launch_t<64, true>(args, chained, st) : launch_t<64, false>(args, chained, st);
}

// Sets every instantiation's shared-memory opt-in (before a stream capture,
// which records launches only).
cudaError_t prepare_launch() {
  cudaError_t e = configure_t<128, false>();
  if (e == cudaSuccess) e = configure_t<128, true>();
  if (e == cudaSuccess) e = configure_t<64, false>();
  if (e == cudaSuccess) e = configure_t<64, true>();
  return e;
}

int smem_bytes() { return kSmemBytes; }

}  // namespace msk
