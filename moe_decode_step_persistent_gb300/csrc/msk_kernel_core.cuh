// Core of the persistent layer kernel: shared-memory plan, per-thread
// context, the bounded grid barrier, the weight-tile schedule shared by the
// producer warp and the compute warps, and the producer itself.
//
// The pages' design ([orcarouter] "Dove si colloca il confine del kernel";
// [ai4snews] "Interpretation"): one resident block per SM with warps whose
// roles are fixed at compile time; one warp loads weights and runs ahead into
// the next operation's weights while the others compute, because weights do
// not depend on the previous operation's output.  Here: warp 8 is that
// producer (bulk copies into a 5-slot shared-memory ring for the dense
// projections and a 4-slot ring of 36 KB stages for the expert GEMMs; warp
// 9 issues the expert GEMMs' tensor-core operations), warps 0..7 compute.
#pragma once

#include "msk_device.cuh"
#include "msk_internal.h"

namespace msk {

// ---------------------------------------------------------------------------
// shared memory plan (dynamic, 232448 bytes available per block)
// ---------------------------------------------------------------------------

struct Misc {
  int abort;
  int n_used;
  int zero;  // always 0: a wait that ignores the abort flag
  int spare;
  uint32_t tmem;  // tensor-memory base address (allocated by warp 0 at launch start)
  uint32_t done_mask;  // expert combine: tokens whose output block this unit completed
  // routing by slot s = t * top_k + r (rank r of token t)
  int slot_e[kMaxT * 8];       // expert
  float slot_gate[kMaxT * 8];  // gate
  uint8_t slot_tok[kMaxT * 8]; // token t
  int used[256];       // used expert ids, ascending
  int ex_start[257];   // by rank in `used`: first position in ex_slots
  uint32_t tok_mask[256];  // by expert id: tokens routed to it (bit t)
  int ex_first[256];   // by expert id: its first position in ex_slots
  uint8_t ex_slots[kMaxT * 8];  // slot ids (t * topk + r) grouped by expert
  int hist[256];
  int pf[32];          // hot experts of the previous step, most used first
  int npf;
  int xq_unit[2];      // expert item queue slots: (g << 16) | (rank << 6) | row block, -1 = no more
  int xq_bcast[2];     // ... as read by compute thread 0, for the other compute threads
  unsigned long long kvmap;  // generic address of the launch's KV tiled-copy map (a kernel parameter)
  float inv_rms[kMaxT];
  float ssq[kMaxT];     // this block's sums of squares of the rows its residual projection wrote
};

constexpr int kOffA = 0;
constexpr int kOffRing = kOffA + kABytes;                      // 131328
constexpr int kOffRed = kOffRing + kSlots * kSlotBytes;        // 213248
constexpr int kRedBytes = 2 * kConsWarps * 32 * 4 * 4;         // 8192
constexpr int kOffBars = kOffRed + kRedBytes;                  // 221440
constexpr int kBarsBytes = 512;
constexpr int kOffMisc = kOffBars + kBarsBytes;
constexpr int kOffArgs = (kOffMisc + (int)sizeof(Misc) + 63) / 64 * 64;  // (LaunchArgs holds a 64-byte aligned map)
constexpr int kSmemBytes = kOffArgs + (int)sizeof(LaunchArgs);
static_assert(kSmemBytes <= 232448, "shared memory plan exceeds the per-block limit");

// During the expert GEMMs the staging area and the ring hold, instead:
// two token-operand buffers (the expert of the block's current and next
// work item: codes in the tensor-core layout, then one scale chunk per MMA), and
// kXSlots weight stages of kUStageBytes that the producer streams and the
// tensor cores consume.
constexpr int kXSlots = 4;
constexpr int kXBBytes = kUN * 2048 / 2 + (2048 / 64) * 512;     // K <= 2048: 16 KB codes + 16 KB chunks
constexpr int kOffXB = 0;
constexpr int kOffXS = kOffXB + 2 * kXBBytes;                     // 65536
static_assert(kOffXS + kXSlots * kUStageBytes <= kOffRed, "expert stages overrun the reduction buffer");
static_assert(kOffXS % 1024 == 0 && kUStageBytes % 1024 == 0, "expert stages are 1 KB aligned");
// tensor memory: kAccs fp32 accumulators of kUN columns per MMA issuer
// (units in flight between the MMA threads and the epilogue warps; issuer i
// accumulates its half of every stage's MMAs at kTmemAcc + i kAccs kUN, the
// epilogues add the halves), then the weights' scale factors per stage
// slot, then the token operands' scale factors
constexpr int kAccs = 4;
constexpr int kTmemCols = 512;
constexpr int kTmemAcc = 0;
constexpr int kAccCols = kMmaIssuers * kAccs * kUN;
// (weight scales per stage slot: kUStageK / 64 MMAs x 4 columns; token
// scales once per expert of the run: up to 32 MMAs x 4 columns each, for at
// most 2 experts)
constexpr int kSfaCols = 4 * (kUStageK / 64);
__device__ __forceinline__ constexpr int tmem_acc(int issuer, int acc) { return kTmemAcc + kUN * (kAccs * issuer + acc); }
__device__ __forceinline__ constexpr int tmem_sfa(int slot, int kk) { return kAccCols + kSfaCols * slot + 4 * kk; }
__device__ __forceinline__ constexpr int tmem_sfb(int j, int jm) { return kAccCols + kSfaCols * kXSlots + 128 * j + 4 * jm; }
static_assert(kAccCols + kSfaCols * kXSlots + 2 * 128 <= kTmemCols, "tensor memory plan exceeds the allocation");

// mbarrier indices
constexpr int BAR_FULL = 0;               // [kSlots] ring slot filled
constexpr int BAR_EMPTY = kSlots;         // [kSlots] ring slot released (8 warps)
constexpr int BAR_XGO = 2 * kSlots;       // routing known: the producer may stream expert stages
constexpr int BAR_HOT = 2 * kSlots + 1;   // router phase reached: time to prefetch the hot experts
constexpr int BAR_STG = 2 * kSlots + 2;   // activation staging landed (one phase per staging)
constexpr int BAR_XFULL = 2 * kSlots + 3;           // [kXSlots] expert weight stage landed
constexpr int BAR_XEMPTY = BAR_XFULL + kXSlots;     // [kXSlots] its MMAs completed (tcgen05.commit of each issuer)
constexpr int BAR_ACCF = BAR_XEMPTY + kXSlots;      // [kAccs] accumulator complete (tcgen05.commit of each issuer)
constexpr int BAR_ACCE = BAR_ACCF + kAccs;          // [kAccs] accumulator read by the 4 epilogue warps
constexpr int BAR_TCDONE = BAR_ACCE + kAccs;        // every tcgen05 operation of the launch completed
// Expert work items are claimed one by one (dynamic); the block's k-th
// item uses queue slot, token-operand buffer and token-scale region k % 2
constexpr int BAR_QFULL = BAR_TCDONE + 1;           // [2] the producer posted the block's next item
constexpr int BAR_QEMPTY = BAR_QFULL + 2;           // [2] ... read by compute thread 0 and the MMA threads
constexpr int BAR_B2RDY = BAR_QEMPTY + 2;           // [2] its token operand is staged
constexpr int BAR_BFREE = BAR_B2RDY + 2;            // [2] its MMAs completed (commit of each issuer): the buffer is free
// The dense phases' activation staging lands in kSegs groups of rows of
// the [16][K] matrix, one barrier each, so that work on the first group
// starts while the later ones stream in
constexpr int kSegs = 4;
constexpr int BAR_SEG = BAR_BFREE + 2;              // [kSegs] staging row group landed
constexpr int BAR_KV = BAR_SEG + kSegs;             // [kAttnStages] attention KV stage landed
constexpr int kNumBars = BAR_KV + kAttnStages;
static_assert(8 * kNumBars <= kBarsBytes, "mbarrier area too small");

// The block's dynamic shared memory (one declaration for every kernel).
extern __shared__ __align__(1024) uint8_t g_smem[];

// Per-thread launch context.  Only the counters that change during the
// launch are stored; everything else is recomputed from special registers or
// read from shared memory (the launch arguments are copied there at launch
// start), so that no phase function touches local memory for them: with
// ~229 KB of shared memory per block the L1 left for local memory is small.
struct Ctx {
  uint32_t seq;     // next ring tile to consume (compute warps) / issue (producer)
  int nbar;         // grid barriers passed in this launch
  unsigned long long bar0;  // grid barrier count at launch start (thread 0 only)
  uint32_t xseq;    // expert weight stages issued (producer) / consumed (MMA thread) in this launch
  uint32_t xunit;   // expert units accumulated (MMA thread) / read back (epilogue warps)
  uint32_t nstg;    // activation stagings waited for (compute threads)
  uint32_t sg;      // activation stagings: 8 x completed + row groups of the current one waited for

  __device__ const LaunchArgs* a() const { return reinterpret_cast<const LaunchArgs*>(g_smem + kOffArgs); }
  __device__ Misc* misc() const { return reinterpret_cast<Misc*>(g_smem + kOffMisc); }
  __device__ uint8_t* smem() const { return g_smem; }
  __device__ uint32_t sbase() const { return smem_u32(g_smem); }
  __device__ int tid() const { return (int)threadIdx.x; }
  __device__ int warp() const { return (int)(threadIdx.x >> 5); }
  __device__ int lane() const { return (int)(threadIdx.x & 31); }
  __device__ int cta() const { return (int)blockIdx.x; }
  __device__ int nctas() const { return (int)gridDim.x; }
  __device__ uint32_t bar(int i) const { return sbase() + kOffBars + 8 * i; }
  __device__ uint32_t slot_addr(int s) const { return sbase() + kOffRing + s * kSlotBytes; }
  __device__ uint32_t xstage(uint32_t n) const { return sbase() + kOffXS + (n % kXSlots) * kUStageBytes; }
  __device__ const volatile int* abort_ptr() const { return &misc()->abort; }
  __device__ uint64_t deadline() const { return gtimer() + a()->budget_ns; }
};

// Copies the launch arguments into shared memory (all threads of the block;
// followed by a block-wide barrier in the caller).  A launch replayed from
// a captured step takes the step's positions and tree from args.step: word
// i of the shared copy is then written once, from there.
__device__ __forceinline__ void stage_args(const LaunchArgs& args) {
  static_assert(sizeof(LaunchArgs) % 4 == 0, "launch arguments are copied as words");
  constexpr int kPos = (int)(offsetof(LaunchArgs, pos0) / 4), kDepth = (int)(offsetof(LaunchArgs, depth) / 4),
                kVis = (int)(offsetof(LaunchArgs, vis) / 4);
  static_assert(kDepth == kPos + 1 && kVis == kDepth + kMaxT, "step fields are contiguous");
  const uint32_t* src = reinterpret_cast<const uint32_t*>(&args);
  uint32_t* dst = reinterpret_cast<uint32_t*>(g_smem + kOffArgs);
  const StepInfo* st = args.step;
  const int vsel = args.cur.window > 0 ? 1 : 0;
  for (int i = threadIdx.x; i < (int)(sizeof(LaunchArgs) / 4); i += blockDim.x) {
    uint32_t v = src[i];
    if (st != nullptr && i >= kPos && i < kVis + kMaxT) {
      if (i == kPos) v = (uint32_t)__ldg(&st->pos0);
      else if (i < kVis) v = (uint32_t)__ldg(&st->depth[i - kDepth]);
      else v = __ldg(&st->vis[vsel][i - kVis]);
    }
    dst[i] = v;
  }
}

constexpr uint32_t ERR_TIMEOUT_BARRIER = 1;
constexpr uint32_t ERR_TIMEOUT_RING = 2;
constexpr uint32_t ERR_TIMEOUT_RING_FREE = 4;  // producer: expert GEMMs never released the ring

// Records a device error (first one wins) and raises the block's abort flag.
__device__ __forceinline__ void raise_error(Ctx& c, uint32_t code, int phase) {
  uint32_t* err = c.a()->s.err;
  if (atomicCAS(err, 0u, code) == 0u) {
    err[1] = (uint32_t)phase;
    err[2] = (uint32_t)c.cta();
  }
  *(volatile int*)&c.misc()->abort = 1;
}

__device__ __forceinline__ bool aborted(const Ctx& c) { return *(volatile int*)&c.misc()->abort != 0; }

// ---------------------------------------------------------------------------
// grid barrier over the compute warps of every block.  One 64-bit counter
// of arrivals that only grows (the host zeroes it after a failed launch):
// a block's arrival is a release reduction that needs no reply, and barrier
// n of a launch is passed once the counter reaches bar0 + n * nctas, where
// bar0 is the count when the launch began.  Every completed launch adds
// nctas arrivals per barrier, so the count is a multiple of nctas between
// launches; a block reading it at launch start may already see up to
// nctas - 1 arrivals of the first barrier (nobody passes that barrier
// before this block arrives), so rounding down gives bar0 exactly.
// Bounded: on expiry the block records ERR_TIMEOUT_BARRIER and every later
// wait returns at once.  Returns false when the launch must stop; the
// decision is taken by thread 0 and published before the closing barrier,
// so all compute threads of a block return the same value.
// ---------------------------------------------------------------------------

__device__ __forceinline__ unsigned long long grid_barrier_base(const unsigned long long* cnt) {
  const unsigned long long v = ld_acquire_gpu_u64(cnt);
  return v - v % (unsigned long long)gridDim.x;
}

static __device__ __noinline__ bool grid_barrier(Ctx& c, int phase) {
  named_bar(1, kConsThreads);
  c.nbar++;
  if (c.tid() == 0) {
    if (!aborted(c)) {
      unsigned long long* cnt = c.a()->s.bar;
      const unsigned long long target = c.bar0 + (unsigned long long)c.nbar * (unsigned long long)c.nctas();
      const bool skip = (c.a()->inject_bar == c.nbar && c.a()->inject_cta == c.cta());
      // release: publishes the block's writes (ordered before it by the
      // named barrier); the acquiring loads below see every arrival's
      if (!skip) red_release_add_gpu_u64(cnt, 1ull);
      const uint64_t dl = c.deadline();
      uint32_t spins = 0;
      while ((long long)(ld_acquire_gpu_u64(cnt) - target) < 0) {
        if ((++spins & 15) == 0) {
          if (ld_relaxed_gpu(c.a()->s.err) != 0u) {
            *(volatile int*)&c.misc()->abort = 1;
            break;
          }
          if (gtimer() > dl) {
            raise_error(c, ERR_TIMEOUT_BARRIER, phase);
            break;
          }
        }
      }
    }
    c.misc()->spare = aborted(c) ? 1 : 0;
  }
  named_bar(1, kConsThreads);
  return *(volatile int*)&c.misc()->spare == 0;
}

__device__ __forceinline__ void stamp(Ctx& c, int slot) {
  if (c.a()->timeline != nullptr && c.tid() == 0)
    c.a()->timeline[(size_t)c.cta() * kTimelineSlots + slot] = gtimer();
}

// ---------------------------------------------------------------------------
// weight tile schedule (identical on producer and compute warps)
// ---------------------------------------------------------------------------

struct DenseSched {
  const uint8_t* base;
  int g0, ng;     // this block's row groups
  int tb, tpg;    // tile bytes, tiles per group
  __device__ int ntiles() const { return ng * tpg; }
};

__device__ __forceinline__ DenseSched dense_sched(const uint8_t* base, int N, int K, int c, int P) {
  DenseSched s;
  const int NG = N / 8;
  s.base = base;
  s.g0 = (int)((long long)c * NG / P);
  s.ng = (int)((long long)(c + 1) * NG / P) - s.g0;
  const int gb = K * 16;
  s.tb = gb < kSlotBytes ? gb : kSlotBytes;
  s.tpg = gb / s.tb;
  return s;
}

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------

// Background prefetch of [p, p + bytes) into L2, one line per lane per
// step over lanes lane0 .. lane0 + nl - 1 of the warp (load/store path).
__device__ __forceinline__ void prefetch_span_lsu(const uint8_t* p, size_t bytes, int lane0, int nl, int lane) {
  if (lane < lane0 || lane >= lane0 + nl) return;
  for (size_t off = (size_t)(lane - lane0) * 128; off < bytes; off += (size_t)nl * 128) prefetch_line_l2(p + off);
}

// A run of one dense projection's tiles (this block's row groups): tile j is
// [first + j tb, first + (j + 1) tb).
struct TileSpan {
  const uint8_t* first;
  int n, tb;
};

__device__ __forceinline__ TileSpan dense_span(const DenseSched s) {
  return TileSpan{s.base + (size_t)s.g0 * s.tpg * s.tb, s.ntiles(), s.tb};
}

// Up to four spans, held in registers (selected by index, no local array).
struct Spans {
  TileSpan s0, s1, s2, s3;
  int n;
  __device__ TileSpan get(int i) const { return i == 0 ? s0 : i == 1 ? s1 : i == 2 ? s2 : s3; }
  __device__ void add(const TileSpan& t) {
    if (n == 0) s0 = t;
    else if (n == 1) s1 = t;
    else if (n == 2) s2 = t;
    else s3 = t;
    ++n;
  }
};

// Streams the spans' tiles, in order, into the ring.  Returns false on abort.
static __device__ __forceinline__ bool produce_spans(Ctx& cin, const Spans& sp, uint64_t policy) {
  Ctx c = cin;  // register copy of the ring position (written back at exit)
  for (int i = 0; i < sp.n; ++i) {
    const TileSpan cs = sp.get(i);
    for (int j = 0; j < cs.n; ++j) {
      const uint32_t s = c.seq % kSlots;
      const uint32_t round = c.seq / kSlots;
      if (c.seq >= (uint32_t)kSlots) {
        if (!mbar_wait(c.bar(BAR_EMPTY + s), (round - 1) & 1, c.deadline(), c.abort_ptr())) {
          if (!aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -1);
          cin = c;
          return false;
        }
      }
      mbar_arrive_expect_tx(c.bar(BAR_FULL + s), (uint32_t)cs.tb);
      bulk_g2s_hint(c.slot_addr(s), cs.first + (size_t)j * cs.tb, (uint32_t)cs.tb, c.bar(BAR_FULL + s), policy);
      c.seq++;
    }
  }
  cin = c;
  return true;
}

// This block's contiguous run [u0, u1) of a GEMM's nunits expert units.
__device__ __forceinline__ void xrun(int nunits, int cta, int nctas, int& u0, int& u1) {
  u0 = (int)((long long)cta * nunits / nctas);
  u1 = (int)((long long)(cta + 1) * nunits / nctas);
}

// One expert unit's weight stages (K order), each one bulk copy into slot
// xseq % kXSlots once the tensor cores have released the slot's previous
// stage.  Returns false on abort or timeout.
static __device__ __forceinline__ bool produce_unit(Ctx& c, const uint8_t* unit, int K, uint64_t pol) {
  const int nst = (K + kUStageK - 1) / kUStageK;
  for (int s = 0; s < nst; ++s) {
    const uint32_t slot = c.xseq % kXSlots;
    if (c.xseq >= (uint32_t)kXSlots &&
        !mbar_wait(c.bar(BAR_XEMPTY + slot), ((c.xseq / kXSlots) - 1) & 1, c.deadline(), c.abort_ptr()))
      return false;
    const uint32_t bytes = (uint32_t)ustage_bytes(ustage_k(K, s));
    mbar_arrive_expect_tx(c.bar(BAR_XFULL + slot), bytes);
    bulk_g2s_hint(c.xstage(c.xseq), unit + (size_t)s * kUStageBytes, bytes, c.bar(BAR_XFULL + slot), pol);
    c.xseq++;
  }
  return true;
}

// Expert work items of a launch, claimed one at a time by the blocks'
// producers from one queue: first every GEMM1 unit (expert rank r, block b
// of I / 64 gate + up row pairs), expert-major, then every GEMM2 unit (rank
// r, block b of P / 128 output rows), numbered in the order in which the
// experts' GEMM1 parts completed (the last GEMM1 epilogue warp of an expert
// appends it to the launch's ready list).  An item is (g << 16) | (r << 6)
// | b; -1: the queue is exhausted; -2: abort or timeout.
constexpr int kItemG = 16, kItemR = 6;
__device__ __forceinline__ int item_g(int it) { return it >> kItemG; }
__device__ __forceinline__ int item_r(int it) { return (it >> kItemR) & 1023; }
__device__ __forceinline__ int item_b(int it) { return it & ((1 << kItemR) - 1); }
static_assert((kMaxK / 64) <= (1 << kItemR) && (kMaxK / kURows) <= (1 << kItemR), "row blocks of an item");

// Queue positions [0, min(GEMM1 units, blocks)) are preassigned: block c's
// first item is position c, known to all its warps as soon as the routing
// is (no claim, no hand-off), so its tensor cores start early.  -4: block c
// has no preassigned item.
__device__ __forceinline__ int first_expert_item(const Ctx& c) {
  const int nbx1 = c.a()->dm.I / 64, n1 = c.misc()->n_used * nbx1;
  return c.cta() < n1 ? (c.cta() / nbx1) << kItemR | (c.cta() % nbx1) : -4;
}

// The next position in the launch's item queue (lane 0 of the producer):
// the claimed positions follow the preassigned ones.
__device__ __forceinline__ uint32_t claim_index(const Ctx& c) {
  const uint32_t n1 = (uint32_t)(c.misc()->n_used * (c.a()->dm.I / 64));
  return min(n1, (uint32_t)c.nctas()) + atomicAdd(c.a()->s.xq + 1, 1u);
}

// True when queue position i resolves without waiting: a GEMM1 item, or
// past the last item.
__device__ __forceinline__ bool claim_is_immediate(const Ctx& c, uint32_t i) {
  const uint32_t nu = (uint32_t)c.misc()->n_used;
  const uint32_t n1 = nu * (uint32_t)(c.a()->dm.I / 64), n2 = nu * (uint32_t)(c.a()->dm.P / kURows);
  return i < n1 || i - n1 >= n2;
}

// The item at queue position i (-1 past the last one, -2 on abort or
// timeout).  A GEMM2 item waits (bounded) until the expert at its
// ready-list position is known.
static __device__ __noinline__ int resolve_item(Ctx& c, uint32_t i) {
  const LaunchArgs& a = *c.a();
  const int nu = c.misc()->n_used, nbx1 = a.dm.I / 64, nbx2 = a.dm.P / kURows;
  const uint32_t n1 = (uint32_t)(nu * nbx1), n2 = (uint32_t)(nu * nbx2);
  if (i < n1) return (int)((i / nbx1) << kItemR | (i % nbx1));
  const uint32_t j = i - n1;
  if (j >= n2) return -1;
  const uint32_t* slot = a.s.xq + 2 + j / nbx2;
  const uint64_t dl = c.deadline();
  uint32_t v, spins = 0;
  while ((v = ld_acquire_gpu(slot)) == 0u) {
    if ((++spins & 15) == 0) {
      if (aborted(c)) return -2;
      if (ld_relaxed_gpu(a.s.err) != 0u) {
        *(volatile int*)&c.misc()->abort = 1;
        return -2;
      }
      if (gtimer() > dl) {
        raise_error(c, ERR_TIMEOUT_BARRIER, PH_GEMM2);
        return -2;
      }
    }
  }
  if (v > (uint32_t)nu) {  // (a rank this block's routing does not have: corrupt queue)
    raise_error(c, ERR_TIMEOUT_RING, PH_GEMM2);
    return -2;
  }
  return (int)(1 << kItemG | (v - 1u) << kItemR | (j % nbx2));
}

// Posts the block's k-th item to slot k % 2 of its item queue, once the
// item two before it was read there.  False on abort or timeout.
__device__ __forceinline__ bool post_item(Ctx& c, uint32_t k, int it) {
  const uint32_t q = k & 1;
  if (k >= 2 && !mbar_wait(c.bar(BAR_QEMPTY + q), ((k >> 1) - 1) & 1, c.deadline(), c.abort_ptr())) return false;
  c.misc()->xq_unit[q] = it;
  mbar_arrive(c.bar(BAR_QFULL + q));  // (release: the slot's value before the arrival)
  return true;
}

// The expert GEMMs' weight stages, in the order the MMA thread consumes
// them: the block's items as it claims them, each posted to the block's
// two-slot item queue (slot k % 2 for the block's k-th item; the sentinel
// -1 ends it) before its stages are issued.  The next item's queue position
// is claimed as soon as an item is posted, and a GEMM1 item (or the end) is
// posted at once: the compute warps can stage its token operand while this
// item's stages stream.  A GEMM2
// item is resolved only after the current item's stages are issued (its
// expert may wait on this very item).  Then waits until every stage has
// been consumed (the stages overlay the ring).  Returns false on abort or
// timeout.
static __device__ __noinline__ bool produce_experts(Ctx& cin, uint64_t pol) {
  Ctx c = cin;
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  Misc* m = c.misc();
  const size_t eb = xexpert_bytes(d.P, d.I);
  bool ok = true;
  int it = first_expert_item(c);
  if (it == -4) it = resolve_item(c, claim_index(c));
  bool posted = false;  // item k is already posted
  for (uint32_t k = 0; ok; ++k) {
    if (it == -2) {
      ok = false;
      break;
    }
    if (!posted && !post_item(c, k, it)) {
      ok = false;
      break;
    }
    if (it < 0) break;
    const uint8_t* ex = a.cur.experts + (size_t)m->used[item_r(it)] * eb;
    const uint8_t* unit = item_g(it) == 0 ? ex + (size_t)item_b(it) * xg1_unit_bytes(d.P)
                                          : ex + xg1_bytes(d.P, d.I) + (size_t)item_b(it) * xg2_unit_bytes(d.I);
    const int K = item_g(it) == 0 ? d.P : d.I;
    const uint32_t ni = claim_index(c);
    int nit = -2;
    posted = claim_is_immediate(c, ni);
    if (posted) {
      nit = resolve_item(c, ni);
      if (!post_item(c, k + 1, nit)) {
        ok = false;
        break;
      }
    }
    ok = produce_unit(c, unit, K, pol);
    if (ok && !posted) nit = resolve_item(c, ni);
    it = nit;
  }
  const uint32_t first = c.xseq > (uint32_t)kXSlots ? c.xseq - kXSlots : 0u;
  for (uint32_t q = first; q < c.xseq && ok; ++q)
    ok = mbar_wait(c.bar(BAR_XEMPTY + q % kXSlots), (q / kXSlots) & 1, c.deadline(), c.abort_ptr());
  if (!ok && !aborted(c)) raise_error(c, ERR_TIMEOUT_RING_FREE, PH_GEMM1);
  cin = c;
  return ok;
}

// Speculative L2 prefetch of the experts the previous step used most
// ([ai4snews] "Interpretation": the 14 most-used experts of the previous
// step's routing are pulled into L2; a wrong guess costs only bandwidth).
// The producer ranks them at launch start (count descending, expert index
// ascending, count > 0); the compute warps issue the prefetch itself late
// in the router phase (prefetch_hot_experts_issue), so that the lines are
// fresh in L2 when the expert GEMMs start.
static __device__ __noinline__ void rank_hot_experts(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  Misc* m = c.misc();
  const int lane = c.lane();
  if (lane == 0) {
    m->npf = 0;
    if (c.cta() == 0) a.s.pf_out[0] = 0;
  }
  if (a.prev_routing == nullptr || d.pf_experts <= 0) return;
  for (int e = lane; e < 256; e += 32) m->hist[e] = 0;
  __syncwarp();
  for (int i = lane; i < d.T * d.topk; i += 32) {
    const int e = __ldcg(a.prev_routing + i);
    if (e >= 0 && e < d.E) atomicAdd(&m->hist[e], 1);
  }
  __syncwarp();
  int npf = 0;
  const int want = min(d.pf_experts, 32);
  for (int r = 0; r < want; ++r) {
    int best_c = 0, best_e = 0x7fffffff;
    for (int e = lane; e < d.E; e += 32) {
      const int cnt = m->hist[e];
      if (cnt > best_c || (cnt == best_c && cnt > 0 && e < best_e)) {
        best_c = cnt;
        best_e = e;
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      const int oc = __shfl_xor_sync(0xffffffffu, best_c, o);
      const int oe = __shfl_xor_sync(0xffffffffu, best_e, o);
      if (oc > best_c || (oc == best_c && oe < best_e)) {
        best_c = oc;
        best_e = oe;
      }
    }
    if (best_c == 0) break;
    if (lane == 0) {
      m->pf[npf] = best_e;
      m->hist[best_e] = 0;
    }
    npf++;
    __syncwarp();
  }
  __syncwarp();
  if (lane == 0) {
    m->npf = npf;
    if (c.cta() == 0) {  // readout for tests (every block ranks the same list)
      a.s.pf_out[0] = npf;
      for (int k = 0; k < npf; ++k) a.s.pf_out[1 + k] = m->pf[k];
    }
  }
}

// This block's share of the ranked hot experts' bytes into L2, issued by
// producer lane 1 when the compute warps reach the router phase, so that
// the lines are fresh in L2 when the expert GEMMs start: a few bulk
// prefetches of at most 64 KB (each a contiguous piece of one expert),
// which the bulk-copy engine works through while the ring is idle (the
// router phase's tiles are already issued), rather than thousands of
// line prefetches, whose stalls would hold up lane 0 of the same warp.
static __device__ __noinline__ void prefetch_hot_experts_issue(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  const Misc* m = c.misc();
  const int npf = m->npf;
  if (npf <= 0) return;
  const size_t eb = xexpert_bytes(d.P, d.I);
  const size_t total = (size_t)npf * eb;
  size_t lo = total * (size_t)c.cta() / c.nctas(), hi = total * (size_t)(c.cta() + 1) / c.nctas();
  lo &= ~(size_t)127;
  hi &= ~(size_t)127;
  while (lo < hi) {
    const int k = (int)(lo / eb);
    const size_t off = lo - (size_t)k * eb, n = min(min(hi - lo, eb - off), (size_t)65536);
    prefetch_l2(a.cur.experts + (size_t)m->pf[k] * eb + off, (uint32_t)n);
    lo += n;
  }
}

// Next layer's cached KV rows (those already in the cache) into L2 near the
// end of this launch ([orcarouter] "Su cosa vengono ancora spesi i 5,9 ms":
// the next launch's old KV rows are prefetched into L2 before it starts).
// Run by the compute warps at the start of the first expert GEMM (while the
// first weight stages stream in), one line per thread per step through the
// load/store path.
static __device__ __noinline__ void prefetch_next_kv(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  if (!a.has_next || a.kv_nxt_ro == nullptr) return;
  const int S = a.pos0;
  int lo = a.nxt.window > 0 ? max(0, S - a.nxt.window + 1) : 0;
  int rows = S - lo;
  if (a.kv_prefetch_rows >= 0 && rows > a.kv_prefetch_rows) {
    lo = S - a.kv_prefetch_rows;
    rows = a.kv_prefetch_rows;
  }
  if (rows <= 0) return;
  const size_t row_b = (size_t)d.hd * 2;
  const size_t blk = (size_t)rows * row_b;     // one (K|V, head) block
  const size_t total = blk * 2 * d.Hkv;
  size_t p0 = total * (size_t)c.cta() / c.nctas(), p1 = total * (size_t)(c.cta() + 1) / c.nctas();
  p0 &= ~(size_t)127;
  p1 &= ~(size_t)127;
  while (p0 < p1) {
    const size_t b = p0 / blk, off = p0 - b * blk;
    const size_t n = min(p1 - p0, blk - off);
    const uint8_t* base = reinterpret_cast<const uint8_t*>(a.kv_nxt_ro) +
                          (b * (size_t)d.max_seq + lo) * row_b + off;
    prefetch_span_lsu(base, n, 0, kConsThreads, c.tid());
    p0 += n;
  }
}

// The producer warp's whole launch.  At launch start the warp ranks the
// previous step's hot experts; lane 1 prefetches them when the compute
// warps reach the router phase.  Then lane 0 streams the dense tiles into the
// ring in the order the compute warps consume them; it runs ahead across
// grid barriers (it never waits on them), bounded only by ring capacity.
// Once the routing is known it streams the expert GEMMs' weight stages
// (which overlay the ring; GEMM2's right after GEMM1's, across the grid
// barrier between them), and after the tensor cores have consumed them it
// fills the ring with the unpool projection's tiles.  The ring's refill at
// the end of each phase is the next phase's head start.
static __device__ void producer(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  const int P = c.nctas();
  const uint64_t pol = policy_evict_first();
  if (aborted(c)) return;  // (an earlier launch of the call failed: nothing to stream)
  rank_hot_experts(c);
  if (c.lane() != 0) {
    if (c.lane() == 1 && mbar_wait(c.bar(BAR_HOT), 0, c.deadline(), c.abort_ptr())) prefetch_hot_experts_issue(c);
    return;
  }
  const int qkv_rows = (d.Hq + 2 * d.Hkv) * d.hd;
  Spans sp;
  sp.n = 0;
  if (a.prologue) sp.add(dense_span(dense_sched(a.cur.w_qkv, qkv_rows, d.D, c.cta(), P)));
  sp.add(dense_span(dense_sched(a.cur.w_o, d.D, d.Hq * d.hd, c.cta(), P)));
  sp.add(dense_span(dense_sched(a.cur.w_pool, d.P, d.D, c.cta(), P)));
  sp.add(dense_span(dense_sched(a.cur.w_router, d.E, d.P, c.cta(), P)));
  bool ok = produce_spans(c, sp, pol);
  // the expert GEMMs' weight stages, once the routing is known (which also
  // means the router phase has consumed every ring tile: the stages overlay
  // the ring)
  if (ok) ok = mbar_wait(c.bar(BAR_XGO), 0, c.deadline(), c.abort_ptr());
  if (ok) ok = produce_experts(c, pol);
  if (ok) {
    sp.n = 0;
    sp.add(dense_span(dense_sched(a.cur.w_unpool, d.D, d.P, c.cta(), P)));
    if (a.has_next) sp.add(dense_span(dense_sched(a.nxt.w_qkv, qkv_rows, d.D, c.cta(), P)));
    ok = produce_spans(c, sp, pol);
  }
  if (!ok) {
    // leave no bulk copy in flight: wait (bounded, ignoring the abort flag)
    // for every ring tile and expert stage issued but possibly not yet landed.
    const volatile int* zero = reinterpret_cast<const volatile int*>(&c.misc()->zero);
    const uint32_t first = c.seq > (uint32_t)kSlots ? c.seq - kSlots : 0u;
    for (uint32_t q = first; q < c.seq; ++q)
      mbar_wait(c.bar(BAR_FULL + q % kSlots), (q / kSlots) & 1, gtimer() + 20000000ull, zero);
    const uint32_t xfirst = c.xseq > (uint32_t)kXSlots ? c.xseq - kXSlots : 0u;
    for (uint32_t q = xfirst; q < c.xseq; ++q)
      mbar_wait(c.bar(BAR_XFULL + q % kXSlots), (q / kXSlots) & 1, gtimer() + 20000000ull, zero);
  }
}

}  // namespace msk
