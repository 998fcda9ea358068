// Core of the persistent layer kernel: shared-memory plan, per-thread
// context, the bounded grid barrier, the weight-tile schedule shared by the
// producer warp and the compute warps, and the producer itself.
//
// The pages' design ([orcarouter] "Dove si colloca il confine del kernel";
// [ai4snews] "Interpretation"): one resident block per SM with warps whose
// roles are fixed at compile time; one warp loads weights and runs ahead into
// the next operation's weights while the others compute, because weights do
// not depend on the previous operation's output.  Here: warp 8 is that
// producer (bulk copies into a 5-slot shared-memory ring plus L2 prefetch of
// the next phase's slice), warps 0..7 compute.
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
  int topk_idx[kMaxT][8];
  float topk_gate[kMaxT][8];
  int used[256];       // used expert ids, ascending
  int ex_start[257];   // by rank in `used`: first position in ex_slots
  int ex_count[256];   // by expert id: number of slots routed to it
  int cursor[256];
  uint8_t ex_slots[kMaxT * 8];  // slot ids (t * topk + r) grouped by expert
  int hist[256];
  int pf[32];
  float inv_rms[kMaxT];
};

constexpr int kOffA = 0;
constexpr int kOffRing = kOffA + kABytes;                      // 131072
constexpr int kOffRed = kOffRing + kSlots * kSlotBytes;        // 212992
constexpr int kRedBytes = 2 * kConsWarps * 32 * 4 * 4;         // 8192
constexpr int kOffBars = kOffRed + kRedBytes;                  // 221184
constexpr int kOffMisc = kOffBars + 128;
constexpr int kSmemBytes = kOffMisc + (int)sizeof(Misc);
static_assert(kSmemBytes <= 232448, "shared memory plan exceeds the per-block limit");

// mbarrier indices
constexpr int BAR_FULL = 0;               // [kSlots] ring slot filled
constexpr int BAR_EMPTY = kSlots;         // [kSlots] ring slot released (8 warps)
constexpr int BAR_KV = 2 * kSlots;        // [2] attention KV stages
constexpr int BAR_DISPATCH = 2 * kSlots + 2;  // routing known (producer waits)

struct Ctx {
  const LaunchArgs* a;
  uint8_t* smem;
  Misc* misc;
  uint32_t sbase;   // shared address of smem
  int cta, nctas;
  int tid, warp, lane;
  uint32_t seq;     // next ring tile to consume (compute warps) / issue (producer)
  int nbar;         // grid barriers passed in this launch

  __device__ uint32_t bar(int i) const { return sbase + kOffBars + 8 * i; }
  __device__ uint32_t slot_addr(int s) const { return sbase + kOffRing + s * kSlotBytes; }
  __device__ const volatile int* abort_ptr() const { return &misc->abort; }
  __device__ uint64_t deadline() const { return gtimer() + a->budget_ns; }
};

constexpr uint32_t ERR_TIMEOUT_BARRIER = 1;
constexpr uint32_t ERR_TIMEOUT_RING = 2;
constexpr uint32_t ERR_TIMEOUT_KV = 3;
constexpr uint32_t ERR_TIMEOUT_DISPATCH = 4;

// Records a device error (first one wins) and raises the block's abort flag.
__device__ __forceinline__ void raise_error(Ctx& c, uint32_t code, int phase) {
  uint32_t* err = c.a->s.err;
  if (atomicCAS(err, 0u, code) == 0u) {
    err[1] = (uint32_t)phase;
    err[2] = (uint32_t)c.cta;
  }
  *(volatile int*)&c.misc->abort = 1;
}

__device__ __forceinline__ bool aborted(const Ctx& c) { return *(volatile int*)&c.misc->abort != 0; }

// ---------------------------------------------------------------------------
// grid barrier over the compute warps of every block (sense by generation;
// self-resetting, so consecutive launches need no host reset).  Bounded: on
// expiry the block records ERR_TIMEOUT_BARRIER and every later wait returns
// at once.  Returns false when the launch must stop; the decision is taken
// by thread 0 and published before the closing barrier, so all compute
// threads of a block return the same value.
// ---------------------------------------------------------------------------

static __device__ bool grid_barrier(Ctx& c, int phase) {
  named_bar(1, kConsThreads);
  c.nbar++;
  if (c.tid == 0) {
    if (!aborted(c)) {
      uint32_t* cnt = c.a->s.bar;
      uint32_t* gen = c.a->s.bar + 1;
      const uint32_t g0 = ld_acquire_gpu(gen);
      const bool skip = (c.a->inject_bar == c.nbar && c.a->inject_cta == c.cta);
      __threadfence();
      bool released = false;
      if (!skip) {
        const uint32_t old = atom_add_acqrel_gpu(cnt, 1u);
        if (old == (uint32_t)c.nctas - 1) {
          st_relaxed_gpu(cnt, 0u);
          red_release_add_gpu(gen, 1u);
          released = true;
        }
      }
      if (!released) {
        const uint64_t dl = c.deadline();
        uint32_t spins = 0;
        while (ld_acquire_gpu(gen) == g0) {
          if ((++spins & 15) == 0) {
            if (ld_relaxed_gpu(c.a->s.err) != 0u) {
              *(volatile int*)&c.misc->abort = 1;
              break;
            }
            if (gtimer() > dl) {
              raise_error(c, ERR_TIMEOUT_BARRIER, phase);
              break;
            }
          }
          __nanosleep(64);
        }
      }
      __threadfence();
    }
    c.misc->spare = aborted(c) ? 1 : 0;
  }
  named_bar(1, kConsThreads);
  return *(volatile int*)&c.misc->spare == 0;
}

__device__ __forceinline__ void stamp(Ctx& c, int slot) {
  if (c.a->timeline != nullptr && c.tid == 0)
    c.a->timeline[(size_t)c.cta * kTimelineSlots + slot] = gtimer();
}

// ---------------------------------------------------------------------------
// weight tile schedule (identical on producer and compute warps)
// ---------------------------------------------------------------------------

struct TileRef {
  const uint8_t* ptr;
  uint32_t bytes;
};

struct DenseSched {
  const uint8_t* base;
  int g0, ng;     // this block's row groups
  int tb, tpg;    // tile bytes, tiles per group
  __device__ int ntiles() const { return ng * tpg; }
  __device__ TileRef tile(const int*, int j) const {
    return TileRef{base + (size_t)(g0 * tpg + j) * tb, (uint32_t)tb};
  }
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

// expert units: unit u of the global list -> (expert, block); tiles of a
// unit in order.
struct ExpertSched {
  const uint8_t* experts;
  size_t eb;         // bytes per expert
  size_t g1b;        // bytes of the GEMM1 region of an expert
  int ublocks;       // blocks per expert (I/16 for GEMM1, P/16 for GEMM2)
  int ubytes;        // bytes per unit
  int nkc;           // k128 chunks per row group
  int tpu;           // tiles per unit
  int u0, nu;        // this block's units
  bool g1;
  __device__ int ntiles() const { return nu * tpu; }
  // tile t of unit u (global unit id)
  __device__ TileRef tile_of(const int* used, int u, int t) const {
    const int e = used[u / ublocks];
    const int b = u % ublocks;
    const uint8_t* ub = experts + (size_t)e * eb + (g1 ? 0 : g1b) + (size_t)b * ubytes;
    if (g1) {
      const int kh = t >> 1, gu = t & 1;
      const int nk = min(8, nkc - 8 * kh);
      return TileRef{ub + (size_t)kh * (2 * 2 * 8 * kBlk4) + (size_t)gu * (2 * nk * kBlk4),
                     (uint32_t)(2 * nk * kBlk4)};
    } else {
      const int kh = t;
      const int nk = min(8, nkc - 8 * kh);
      return TileRef{ub + (size_t)kh * (2 * 8 * kBlk4), (uint32_t)(2 * nk * kBlk4)};
    }
  }
  __device__ TileRef tile(const int* used, int j) const { return tile_of(used, u0 + j / tpu, j % tpu); }
};

__device__ __forceinline__ ExpertSched expert_sched(const LaunchArgs& a, const LayerDev& L, int n_used,
                                                    bool g1, int c, int P) {
  const Dims& d = a.dm;
  ExpertSched s;
  s.experts = L.experts;
  s.eb = expert_bytes(d.P, d.I);
  s.g1b = expert_g1_bytes(d.P, d.I);
  s.g1 = g1;
  if (g1) {
    s.ublocks = d.I / 16;
    s.ubytes = g1_unit_bytes(d.P);
    s.nkc = d.P / 128;
    s.tpu = 2 * ((s.nkc + 7) / 8);
  } else {
    s.ublocks = d.P / 16;
    s.ubytes = g2_unit_bytes(d.I);
    s.nkc = d.I / 128;
    s.tpu = (s.nkc + 7) / 8;
  }
  const long long NU = (long long)n_used * s.ublocks;
  s.u0 = (int)(c * NU / P);
  s.nu = (int)((c + 1) * NU / P) - s.u0;
  return s;
}

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------

// Prefetches [p, p + bytes) into L2 in 32 KB pieces (16-byte granularity).
__device__ __forceinline__ void prefetch_bytes(const uint8_t* p, size_t bytes) {
  const uint8_t* end = p + (bytes & ~(size_t)15);
  while (p < end) {
    const size_t n = (size_t)(end - p) < 32768 ? (size_t)(end - p) : 32768;
    prefetch_l2(p, (uint32_t)n);
    p += n;
  }
}

__device__ __forceinline__ void prefetch_dense_slice(const DenseSched& s) {
  if (s.ng > 0) prefetch_bytes(s.base + (size_t)s.g0 * s.tpg * s.tb, (size_t)s.ng * s.tpg * s.tb);
}

// Streams `n` tiles into the ring.  Returns false on abort.
template <class Sched>
static __device__ bool produce_tiles(Ctx& c, const Sched& sch, const int* used, int n, uint64_t policy) {
  for (int j = 0; j < n; ++j) {
    const uint32_t s = c.seq % kSlots;
    const uint32_t round = c.seq / kSlots;
    if (c.seq >= (uint32_t)kSlots) {
      if (!mbar_wait(c.bar(BAR_EMPTY + s), (round - 1) & 1, c.deadline(), c.abort_ptr())) {
        if (!aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -1);
        return false;
      }
    }
    const TileRef t = sch.tile(used, j);
    mbar_arrive_expect_tx(c.bar(BAR_FULL + s), t.bytes);
    bulk_g2s_hint(c.slot_addr(s), t.ptr, t.bytes, c.bar(BAR_FULL + s), policy);
    c.seq++;
  }
  return true;
}

// Speculative L2 prefetch of the experts the previous step used most
// ([ai4snews] "Interpretation": the 14 most-used experts of the previous
// step's routing are pulled into L2; a wrong guess costs only bandwidth).
// Ranked by count descending, expert index ascending, count > 0.  Every
// producer lane takes part in the ranking; each block prefetches its share
// of the chosen experts' bytes.
static __device__ void prefetch_hot_experts(Ctx& c) {
  const LaunchArgs& a = *c.a;
  const Dims& d = a.dm;
  Misc* m = c.misc;
  const int lane = c.lane;
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
  if (lane == 0 && npf > 0) {
    const size_t eb = expert_bytes(d.P, d.I);
    const size_t total = (size_t)npf * eb;
    size_t lo = total * (size_t)c.cta / c.nctas, hi = total * (size_t)(c.cta + 1) / c.nctas;
    lo &= ~(size_t)15;
    hi &= ~(size_t)15;
    while (lo < hi) {
      const int k = (int)(lo / eb);
      const size_t off = lo - (size_t)k * eb;
      const size_t n = min(hi - lo, eb - off);
      prefetch_bytes(a.cur.experts + (size_t)m->pf[k] * eb + off, n);
      lo += n;
    }
  }
  __syncwarp();
}

// Next layer's cached KV rows (those already in the cache) into L2 near the
// end of this launch ([orcarouter] "Su cosa vengono ancora spesi i 5,9 ms":
// the next launch's old KV rows are prefetched into L2 before it starts).
static __device__ void prefetch_next_kv(Ctx& c) {
  const LaunchArgs& a = *c.a;
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
  size_t p0 = total * (size_t)c.cta / c.nctas, p1 = total * (size_t)(c.cta + 1) / c.nctas;
  p0 &= ~(size_t)15;
  p1 &= ~(size_t)15;
  while (p0 < p1) {
    const size_t b = p0 / blk, off = p0 - b * blk;
    const size_t n = min(p1 - p0, blk - off);
    const uint8_t* base = reinterpret_cast<const uint8_t*>(a.kv_nxt_ro) +
                          (b * (size_t)d.max_seq + lo) * row_b + off;
    prefetch_bytes(base, n);
    p0 += n;
  }
}

// The producer's whole launch: the same tile order the compute warps
// consume.  Runs ahead across grid barriers (it never waits on them), bounded
// only by ring capacity, and by the routing for the expert phases.
static __device__ void producer(Ctx& c) {
  const LaunchArgs& a = *c.a;
  const Dims& d = a.dm;
  const int P = c.nctas;
  const uint64_t pol = policy_evict_first();
  prefetch_hot_experts(c);
  if (c.lane != 0) return;
  const DenseSched s_pro = dense_sched(a.cur.w_qkv, (d.Hq + 2 * d.Hkv) * d.hd, d.D, c.cta, P);
  const DenseSched s_o = dense_sched(a.cur.w_o, d.D, d.Hq * d.hd, c.cta, P);
  const DenseSched s_pool = dense_sched(a.cur.w_pool, d.P, d.D, c.cta, P);
  const DenseSched s_r = dense_sched(a.cur.w_router, d.E, d.P, c.cta, P);
  const DenseSched s_un = dense_sched(a.cur.w_unpool, d.D, d.P, c.cta, P);
  const DenseSched s_qkv = dense_sched(a.nxt.w_qkv, (d.Hq + 2 * d.Hkv) * d.hd, d.D, c.cta, P);
  bool ok = true;
  prefetch_dense_slice(s_o);
  if (a.prologue) ok = produce_tiles(c, s_pro, nullptr, s_pro.ntiles(), pol);
  if (ok) {
    prefetch_dense_slice(s_pool);
    ok = produce_tiles(c, s_o, nullptr, s_o.ntiles(), pol);
  }
  if (ok) {
    prefetch_dense_slice(s_r);
    ok = produce_tiles(c, s_pool, nullptr, s_pool.ntiles(), pol);
  }
  if (ok) ok = produce_tiles(c, s_r, nullptr, s_r.ntiles(), pol);
  if (ok) {
    // expert tiles need the routing of this step
    if (!mbar_wait(c.bar(BAR_DISPATCH), 0, c.deadline(), c.abort_ptr())) {
      if (!aborted(c)) raise_error(c, ERR_TIMEOUT_DISPATCH, PH_TOPK);
      ok = false;
    }
  }
  if (ok) {
    const int nu = c.misc->n_used;
    const ExpertSched g1 = expert_sched(a, a.cur, nu, true, c.cta, P);
    const ExpertSched g2 = expert_sched(a, a.cur, nu, false, c.cta, P);
    // this block's GEMM2 units into L2 while GEMM1 streams
    for (int u = g2.u0; u < g2.u0 + g2.nu; ++u) {
      const TileRef t = g2.tile_of(c.misc->used, u, 0);
      prefetch_bytes(t.ptr, (size_t)g2.ubytes);
    }
    ok = produce_tiles(c, g1, c.misc->used, g1.ntiles(), pol);
    if (ok) {
      prefetch_dense_slice(s_un);
      ok = produce_tiles(c, g2, c.misc->used, g2.ntiles(), pol);
    }
  }
  if (ok) {
    if (a.has_next) prefetch_dense_slice(s_qkv);
    prefetch_next_kv(c);
    ok = produce_tiles(c, s_un, nullptr, s_un.ntiles(), pol);
  }
  if (ok && a.has_next) ok = produce_tiles(c, s_qkv, nullptr, s_qkv.ntiles(), pol);
  if (!ok) {
    // leave no bulk copy in flight: wait (bounded, ignoring the abort flag)
    // for every tile issued but possibly not yet landed.
    const uint32_t first = c.seq > (uint32_t)kSlots ? c.seq - kSlots : 0u;
    for (uint32_t q = first; q < c.seq; ++q)
      mbar_wait(c.bar(BAR_FULL + q % kSlots), (q / kSlots) & 1, gtimer() + 20000000ull,
                reinterpret_cast<const volatile int*>(&c.misc->zero));
  }
}

}  // namespace msk
