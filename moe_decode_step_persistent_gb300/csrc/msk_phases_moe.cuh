// Compute-warp phases, part 2: router top-k and dispatch, the NVFP4 expert
// GEMMs, and the gated combine of expert outputs.
//
// Expert numerics follow the pages: expert weights in NVFP4 ([newruntime]
// "What happened"), the first expert GEMM's output quantised to fp4 and the
// second's kept in bf16 ([orcarouter] "Dove si colloca il confine del
// kernel").  Both GEMM inputs are NVFP4 (W4A4).  Codes times block scales
// are exact in fp16, so the tensor cores see exactly the dequantised values
// and accumulate in fp32; tensor scales are applied to the fp32 sums.
#pragma once

#include "msk_phases_dense.cuh"

namespace msk {

// ---------------------------------------------------------------------------
// router: top-k per token (logit descending, index ascending), softmax over
// the selected logits; then dispatch lists, identical in every block.
// ---------------------------------------------------------------------------

static_assert(kMaxT * 8 <= 4 * 32, "dispatch handles at most four rounds of 32 slots");
static __device__ __noinline__ void topk_dispatch(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  Misc* m = c.misc();
  // each half-warp ranks one token (t = 2 w + half): lane hl of the half
  // holds candidates hl + 16 j as 64-bit keys (order-preserving logit bits
  // above, 0xFFFF - expert below: the larger key is the larger logit, ties
  // to the smaller expert index; 0 = no candidate).  A round takes the
  // lane's best key and the half-warp's best by 4 shuffle levels, and
  // retires it.  After round r, lane r of the half holds the r-th choice.
  static_assert(kMaxT <= 2 * kConsWarps, "one token per half-warp");
  const int hl = c.lane() & 15, hbase = c.lane() & 16;
  const int t = 2 * c.warp() + (c.lane() >> 4);
  const bool live = t < d.T;
  uint64_t key[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int e = hl + 16 * j;
    key[j] = 0;
    if (live && e < d.E) {
      const uint32_t b = __float_as_uint(__ldcg(a.s.logits + (size_t)t * d.E + e));
      const uint32_t ob = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
      key[j] = ((uint64_t)ob << 32) | (uint32_t)(0xFFFF - e);
    }
  }
  stamp(c, 30);
  uint64_t mine = 0;
#pragma unroll 1
  for (int r = 0; r < d.topk; ++r) {
    uint64_t best = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    // keys are unique (the expert index is part of the key): retire the winner
#pragma unroll
    for (int j = 0; j < 16; ++j) key[j] = key[j] == best ? 0 : key[j];
    if (hl == r) mine = best;
  }
  const uint32_t mob = (uint32_t)(mine >> 32);
  const float my_v = mine == 0 ? -CUDART_INF_F : __uint_as_float((mob & 0x80000000u) ? (mob & 0x7FFFFFFFu) : ~mob);
  const int my_e = mine == 0 ? 0 : 0xFFFF - (int)(mine & 0xFFFFu);
  stamp(c, 31);
  // softmax over the selected logits: lane r's exp, summed in rank order
  {
    const float top = __shfl_sync(0xffffffffu, my_v, hbase);
    const float ex = hl < d.topk ? expf(my_v - top) : 0.f;
    float sum = 0.f;
    for (int r = 0; r < d.topk; ++r) sum += __shfl_sync(0xffffffffu, ex, hbase + r);
    if (live && hl < d.topk) {
      m->topk_idx[t][hl] = my_e;
      m->topk_gate[t][hl] = ex / sum;
    }
  }
  named_bar(1, kConsThreads);
  stamp(c, 14);  // top-k chosen (timing builds only: stamp is a no-op without a timeline)
  if (c.cta() == 0 && a.routing_out != nullptr)
    for (int i = c.tid(); i < d.T * d.topk; i += kConsThreads) a.routing_out[i] = m->topk_idx[i / d.topk][i % d.topk];
  if (c.warp() == 0) {
    // slots s = t k + r in rounds of 32: per round, lanes holding the same
    // expert form a match group; its lowest lane adds the group's size
    const int nslots = d.T * d.topk;
    for (int e = c.lane(); e < 256; e += 32) m->ex_count[e] = 0;
    __syncwarp();
    unsigned grp[4];
    int ex[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int s = 32 * q + c.lane();
      ex[q] = s < nslots ? m->topk_idx[s / d.topk][s % d.topk] : -1 - c.lane();
      grp[q] = __match_any_sync(0xffffffffu, ex[q]);
      if (s < nslots && (grp[q] & ((1u << c.lane()) - 1u)) == 0u) m->ex_count[ex[q]] += __popc(grp[q]);
      __syncwarp();
    }
    // lane l owns experts [8l, 8l + 8): ranks and slot offsets by warp scans
    int nu = 0, ns = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int cnt = m->ex_count[8 * c.lane() + j];
      nu += cnt > 0;
      ns += cnt;
    }
    int nu_x = nu, ns_x = ns;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a1 = __shfl_up_sync(0xffffffffu, nu_x, o), a2 = __shfl_up_sync(0xffffffffu, ns_x, o);
      if (c.lane() >= o) {
        nu_x += a1;
        ns_x += a2;
      }
    }
    int rank = nu_x - nu, start = ns_x - ns;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 8 * c.lane() + j;
      const int cnt = m->ex_count[e];
      if (cnt > 0) {
        m->used[rank] = e;
        m->ex_start[rank] = start;
        m->cursor[e] = start;
        rank++;
        start += cnt;
      }
    }
    if (c.lane() == 31) {
      m->n_used = nu_x;
      m->ex_start[nu_x] = ns_x;
    }
    __syncwarp();
    // slots grouped by expert, ascending slot order inside a group
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int s = 32 * q + c.lane();
      const int rk = __popc(grp[q] & ((1u << c.lane()) - 1u));
      int base = 0;
      if (s < nslots) base = m->cursor[ex[q]];
      __syncwarp();
      if (s < nslots) {
        m->ex_slots[base + rk] = (uint8_t)s;
        if (rk == 0) m->cursor[ex[q]] = base + __popc(grp[q]);
      }
      __syncwarp();
    }
  }
  named_bar(1, kConsThreads);
  stamp(c, 15);  // dispatch lists ready
}

// ---------------------------------------------------------------------------
// NVFP4 helpers
// ---------------------------------------------------------------------------

// One 576-byte weight block (8 rows x k128) as one lane holds it: its 16
// bytes of codes (two E2M1 per byte, in mma fragment order) and the 8 E4M3
// scales of its row g = lane / 4.
struct Fp4Blk {
  uint4 c;
  uint2 s;
};

// Weight bytes are used once per launch: read around L1 and mark them
// first in line for L2 eviction.
__device__ __forceinline__ uint4 ldg_stream16(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

__device__ __forceinline__ uint2 ldg_stream8(const void* p, uint64_t pol) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
               : "=r"(r.x), "=r"(r.y)
               : "l"(p), "l"(pol));
  return r;
}

__device__ __forceinline__ Fp4Blk ld_blk(const uint8_t* blk, int lane, uint64_t pol) {
  Fp4Blk b;
  b.c = ldg_stream16(blk + lane * 16, pol);
  b.s = ldg_stream8(blk + 512 + (lane >> 2) * 8, pol);
  return b;
}

// acc += A (16 x k128, f16 fragments in `af`) times one weight block held
// in registers, dequantised on the fly (E2M1 x E4M3 is exact in fp16): the
// 8 scales are converted pairwise once, each k16 step takes its scale as a
// broadcast half, and code bytes go straight from the word into the cvt.
__device__ __forceinline__ void fp4_blk_mma(float (&acc)[4], const uint32_t (&af)[8][4], const Fp4Blk& b) {
  const uint32_t cws[4] = {b.c.x, b.c.y, b.c.z, b.c.w};
  const uint32_t sp[4] = {e4m3_pair_to_f16x2(b.s.x, 0), e4m3_pair_to_f16x2(b.s.x, 1), e4m3_pair_to_f16x2(b.s.y, 0),
                          e4m3_pair_to_f16x2(b.s.y, 1)};
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t scf = f16x2_bcast(sp[s >> 1], s & 1);
    const uint32_t b0 = hmul2(e2m1_byte_to_f16x2(cws[s >> 1], 2 * (s & 1)), scf);
    const uint32_t b1 = hmul2(e2m1_byte_to_f16x2(cws[s >> 1], 2 * (s & 1) + 1), scf);
    mma_f16(acc, af[s], b0, b1);
  }
}

// The same for a block in shared memory.
__device__ __forceinline__ void fp4_block_mma(float (&acc)[4], const uint32_t (&af)[8][4], uint32_t blk, int lane) {
  Fp4Blk b;
  b.c = lds128(blk + lane * 16);
  b.s = lds64(blk + 512 + (lane >> 2) * 8);
  fp4_blk_mma(acc, af, b);
}

// A fragments (8 k16 steps of a k128 chunk) from a gathered [rows][K] f16
// matrix in the staging area: fragment row i reads physical row prow.
__device__ __forceinline__ void load_a_chunk(uint32_t (&af)[8][4], uint32_t A, int prow, int K, int kc,
                                             int lane) {
  const uint32_t rb_ = A + prow * (K * 2);
  const int sw = prow & 7;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int ch = ((kc * 128 + 16 * s) >> 3) + (lane >> 4);
    ldmatrix_x4(af[s], rb_ + ((ch ^ sw) << 4));
  }
}

// Q4 of 16 fp32 values held 4 per lane across the 4 lanes of a quad
// (rows {2c, 2c+1, 8+2c, 9+2c} for lane c): E4M3 scale of amax / 6, E2M1
// codes of x / scale, both round-to-nearest-even with saturation.
struct Q4Out {
  uint32_t byte_lo, byte_hi, scale;
};
__device__ __forceinline__ Q4Out q4_quad(const float (&x)[4]) {
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  Q4Out r{0u, 0u, 0u};
  if (amax == 0.f) return r;
  const uint32_t sc = f32_to_e4m3(amax / 6.0f);
  const float dec = e4m3_to_f32(sc);
  r.scale = sc;
  if (dec == 0.f) return r;
  r.byte_lo = f32x2_to_e2m1x2(x[0] / dec, x[1] / dec);
  r.byte_hi = f32x2_to_e2m1x2(x[2] / dec, x[3] / dec);
  return r;
}

// Units a warp's L2 prefetch runs ahead of the unit it streams (GEMM1;
// GEMM2's units are a quarter the size and run twice as far ahead).
constexpr int kUnitsAhead = 1;

// The expert units (expert in rank order, then row block) of a GEMM are
// split into contiguous runs, one per compute warp of the grid; a warp owns
// its units outright (whole K), so no cross-warp reduction is needed.
__device__ __forceinline__ void warp_run(int nunits, const Ctx& c, int& u0, int& u1) {
  const long long nw = (long long)c.nctas() * kConsWarps, gw = (long long)c.cta() * kConsWarps + c.warp();
  u0 = (int)(gw * nunits / nw);
  u1 = (int)((gw + 1) * nunits / nw);
}

// ---------------------------------------------------------------------------
// Q4 of the pooled activations, once per launch: each block quantises its
// share of the (token, 16-block) items from the pooled rows it has staged
// for the router and writes the dequantised f16 values for every block's
// GEMM1.
// ---------------------------------------------------------------------------

static __device__ __noinline__ void quantize_pooled(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  const int P = d.P, per = P / 16, n = d.T * per;
  const uint8_t* Ag = c.smem() + kOffA;
  const int i0 = (int)((long long)c.cta() * n / c.nctas()), i1 = (int)((long long)(c.cta() + 1) * n / c.nctas());
  for (int q = i0 + c.tid(); q < i1; q += kConsThreads) {
    const int t = q / per, blk = q % per;
    const uint4 v0 = *reinterpret_cast<const uint4*>(Ag + a_chunk_off(t, 2 * blk, P));
    const uint4 v1 = *reinterpret_cast<const uint4*>(Ag + a_chunk_off(t, 2 * blk + 1, P));
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t out[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float x[16];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      x[2 * j] = bf16_lo(w[j]);
      x[2 * j + 1] = bf16_hi(w[j]);
      amax = fmaxf(amax, fmaxf(fabsf(x[2 * j]), fabsf(x[2 * j + 1])));
    }
    if (amax > 0.f) {
      const uint32_t sc = f32_to_e4m3(amax / 6.0f);
      const float dec = e4m3_to_f32(sc);
      if (dec > 0.f) {
        const uint32_t scf = e4m3x2_to_f16x2(sc | (sc << 8));
#pragma unroll
        for (int j = 0; j < 8; ++j)
          out[j] = hmul2(e2m1x2_to_f16x2(f32x2_to_e2m1x2(x[2 * j] / dec, x[2 * j + 1] / dec)), scf);
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(a.s.a4 + (size_t)t * P + 16 * blk);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  }
}

// ---------------------------------------------------------------------------
// Per-warp weight streaming for the expert GEMMs: a warp's steps go through
// its kXStages private stages, kXStages - 1 in flight ahead of the one being
// multiplied (bulk copies completing on the stage's mbarrier).  Waits are
// bounded; on expiry the warp drains what it issued and reports false.
// ---------------------------------------------------------------------------

__device__ __forceinline__ bool xstage_wait(Ctx& c) {
  const bool got = mbar_wait(c.xbar(c.xs_done), (c.xs_done / kXStages) & 1, c.deadline(), c.abort_ptr());
  const bool ok = __all_sync(0xffffffffu, got);
  if (!ok && c.lane() == 0 && !aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -3);
  return ok;
}

// Lets every copy this warp issued land before the block may exit.
__device__ __forceinline__ void xstage_drain(Ctx& c) {
  const uint64_t dl = c.deadline();
  while (c.xs_done < c.xs_issued) {
    mbar_wait(c.xbar(c.xs_done), (c.xs_done / kXStages) & 1, dl, &c.misc()->zero);
    c.xs_done++;
  }
  __syncwarp();
}

// This warp's GEMM2 weight stream: its run of units (expert rank, 16 output
// rows) and the steps of four k128 chunks (8 blocks, one contiguous range)
// they are streamed in.
struct G2Stream {
  int ub, ubytes, nkc, spu, u0, u1, nsteps;
  size_t eb, g1b;
};

__device__ __forceinline__ G2Stream g2_stream(const Ctx& c) {
  const Dims& d = c.a()->dm;
  G2Stream s;
  s.ub = d.P / 16;
  warp_run(c.misc()->n_used * s.ub, c, s.u0, s.u1);
  s.ubytes = g2_unit_bytes(d.I);
  s.nkc = d.I / 128;
  s.spu = (s.nkc + 3) / 4;
  s.nsteps = (s.u1 - s.u0) * s.spu;
  s.eb = expert_bytes(d.P, d.I);
  s.g1b = expert_g1_bytes(d.P, d.I);
  return s;
}

__device__ __forceinline__ const uint8_t* g2_unit_ptr(const Ctx& c, const G2Stream& s, int u) {
  return c.a()->cur.experts + (size_t)c.misc()->used[u / s.ub] * s.eb + s.g1b + (size_t)(u % s.ub) * s.ubytes;
}

// Issues step j of the stream into this warp's next stage.
__device__ __forceinline__ void g2_issue(Ctx& c, const G2Stream& s, int j, uint64_t pol) {
  if (c.lane() == 0) {
    const int kc0 = 4 * (j % s.spu), nb = min(4, s.nkc - kc0);
    const uint32_t bar = c.xbar(c.xs_issued);
    mbar_arrive_expect_tx(bar, 2 * nb * kBlk4);
    bulk_g2s_hint(c.xstage(c.xs_issued), g2_unit_ptr(c, s, s.u0 + j / s.spu) + g2_blk_off(kc0, 0), 2 * nb * kBlk4, bar,
                  pol);
  }
  c.xs_issued++;
}

__device__ __forceinline__ void g2_prefetch_unit(const Ctx& c, const G2Stream& s, int u, uint64_t pol) {
  if (c.lane() == 0 && u < s.u1) prefetch_l2_hint(g2_unit_ptr(c, s, u), (uint32_t)s.ubytes, pol);
}

// ---------------------------------------------------------------------------
// expert GEMM1 (+ SwiGLU + Q4): unit = (expert, 16 intermediate rows),
// gate and up together, whole K
// ---------------------------------------------------------------------------

static __device__ __noinline__ void gemm1_phase(Ctx& cin) {
  Ctx c = cin;  // register copy of the stage counters (written back at exit)
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  Misc* m = c.misc();
  const int P = d.P;
  uint8_t* Ag = c.smem() + kOffA;
  const uint32_t A = c.sbase() + kOffA;
  const int ub = d.I / 16;  // units per expert
  int u0, u1;
  warp_run(m->n_used * ub, c, u0, u1);
  const size_t eb = expert_bytes(P, d.I);
  const int ubytes = g1_unit_bytes(P);
  const uint8_t* experts = a.cur.experts;
  auto unit_ptr = [&](int u) -> const uint8_t* {
    return experts + (size_t)m->used[u / ub] * eb + (size_t)(u % ub) * ubytes;
  };
  const uint64_t pol = policy_evict_first();
  const int nkc = P / 128;
  const int spu = (nkc + 1) / 2;  // steps (two k128 chunks, 8 blocks) per unit
  const int nsteps = (u1 - u0) * spu;
  // step j = chunks kc0, kc0 + 1 of its unit: one contiguous range, block
  // (chunk kc0 + h, gate/up gu, row group gr) at 4 h + 2 gu + gr
  auto issue_step = [&](int j) {
    if (c.lane() == 0) {
      const int kc0 = 2 * (j % spu), nb = min(2, nkc - kc0);
      const uint32_t bar = c.xbar(c.xs_issued);
      mbar_arrive_expect_tx(bar, 4 * nb * kBlk4);
      bulk_g2s_hint(c.xstage(c.xs_issued), unit_ptr(u0 + j / spu) + g1_blk_off(kc0, 0, 0), 4 * nb * kBlk4, bar, pol);
    }
    c.xs_issued++;
  };
  // whole units into L2 (two 18 KB halves), kUnitsAhead ahead of the one
  // being streamed
  auto prefetch_unit = [&](int u) {
    if (c.lane() < 2 && u < u1) prefetch_l2_hint(unit_ptr(u) + c.lane() * (ubytes / 2), (uint32_t)(ubytes / 2), pol);
  };
  // a = Q4(pooled) dequantised (f16 [17][P], row 16 = zeros); its copies
  // go out ahead of the weight requests so they are not queued behind them
  stage_issue(cin, a.s.a4, P);
  for (int q = c.tid(); q < P / 8; q += kConsThreads)
    *reinterpret_cast<uint4*>(Ag + a_chunk_off(16, q, P)) = make_uint4(0, 0, 0, 0);
  // the warp's first steps: in flight while the activations land
  for (int j = 0; j < kXStages - 1 && j < nsteps; ++j) issue_step(j);
  for (int k = 0; k <= kUnitsAhead; ++k) prefetch_unit(u0 + k);
  cp_async_wait_all();
  named_bar(1, kConsThreads);
  stamp(c, kSlotExpert + 0);

  const int g = c.lane() >> 2, cq = c.lane() & 3;
  float acc[2][2][4];
  int prow = 16, b = 0, st = 0, ne = 0;
  float tsg = 0.f, tsu = 0.f;
#pragma unroll 1
  for (int j = 0; j < nsteps; ++j) {
    const int kc0 = 2 * (j % spu);
    if (kc0 == 0) {
      const int u = u0 + j / spu;
      const int rank = u / ub;
      const int e = m->used[rank];
      b = u % ub;
      st = m->ex_start[rank];
      ne = m->ex_start[rank + 1] - st;
      const int fi = c.lane() & 15;
      prow = fi < ne ? m->ex_slots[st + fi] / d.topk : 16;
      tsg = __ldg(a.cur.ts + 3 * e);
      tsu = __ldg(a.cur.ts + 3 * e + 1);
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 2; ++y) acc[x][y][0] = acc[x][y][1] = acc[x][y][2] = acc[x][y][3] = 0.f;
      if (j > 0) prefetch_unit(u + kUnitsAhead);
    }
    if (j + kXStages - 1 < nsteps) issue_step(j + kXStages - 1);
    if (!xstage_wait(c)) break;
    const uint32_t stage = c.xstage(c.xs_done);
#pragma unroll 1
    for (int h = 0; h < 2; ++h)
      if (kc0 + h < nkc) {
        uint32_t af[8][4];
        load_a_chunk(af, A, prow, P, kc0 + h, c.lane());
#pragma unroll
        for (int q = 0; q < 4; ++q) fp4_block_mma(acc[q >> 1][q & 1], af, stage + (4 * h + q) * kBlk4, c.lane());
      }
    __syncwarp();
    c.xs_done++;
    if (kc0 + 2 >= nkc) {
      // SwiGLU of this unit's 16 rows, then Q4 per (slot, 16-block):
      // acc[0] gate, acc[1] up; [gr] rows 8 gr + {2c, 2c+1}; [0,1] slot g, [2,3] slot g+8
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float s[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int gr = jj >> 1, k = 2 * hh + (jj & 1);
          const float gv = acc[0][gr][k] * tsg, uv = acc[1][gr][k] * tsu;
          s[jj] = gv / (1.0f + expf(-gv)) * uv;
        }
        const Q4Out q = q4_quad(s);
        const int fi2 = g + 8 * hh;
        if (fi2 < ne) {
          const int slot = m->ex_slots[st + fi2];
          uint8_t* codes = a.s.sq_codes + (size_t)slot * (d.I / 2);
          codes[8 * b + cq] = (uint8_t)q.byte_lo;
          codes[8 * b + 4 + cq] = (uint8_t)q.byte_hi;
          if (cq == 0) a.s.sq_scales[(size_t)slot * (d.I / 16) + b] = (uint8_t)q.scale;
        }
      }
    }
    if (j == 0) stamp(c, kSlotExpert + 1);
  }
  xstage_drain(c);
  stamp(c, kSlotExpert + 2);
  if (!aborted(c)) {
    // head start for GEMM2 (its weights do not depend on GEMM1): this
    // warp's first steps stream in while the grid waits at the barrier
    const G2Stream s2 = g2_stream(c);
    for (int j = 0; j < kXStages - 1 && j < s2.nsteps; ++j) g2_issue(c, s2, j, pol);
    for (int k = 0; k <= 2 * kUnitsAhead; ++k) g2_prefetch_unit(c, s2, s2.u0 + k, pol);
  }
  cin = c;
}

// ---------------------------------------------------------------------------
// expert GEMM2: unit = (expert, 16 output rows); y = rb(s_q W_down^T), then
// the gated combine m[t] = rb(sum_r gate[t][r] y[t k + r]) (rank order) by
// whichever unit completes a (token, 16-row block) last
// ---------------------------------------------------------------------------

static __device__ __noinline__ void gemm2_phase(Ctx& cin) {
  Ctx c = cin;  // register copy of the stage counters (written back at exit)
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  Misc* m = c.misc();
  const int I = d.I, P = d.P;
  uint8_t* Ag = c.smem() + kOffA;
  const uint32_t A = c.sbase() + kOffA;
  const G2Stream s2 = g2_stream(c);
  const int ub = s2.ub, nkc = s2.nkc, spu = s2.spu, nsteps = s2.nsteps, u0 = s2.u0;
  const int nunits = m->n_used * ub;
  const uint64_t pol = policy_evict_first();
  // steps already issued at the end of GEMM1
  const int pre = (int)(c.xs_issued - c.xs_done);
  auto issue_step = [&](int j) { g2_issue(c, s2, j, pol); };

  // The block's units span at most two experts (its share of the unit list
  // is at most one expert's worth, checked at model creation).  Stage their
  // slots' fp4 intermediates dequantised to f16: rows 16 j + i for the i-th
  // slot of the block's j-th expert; row 32 is zeros.
  const long long nw = (long long)c.nctas() * kConsWarps;
  const int cu0 = (int)((long long)c.cta() * kConsWarps * nunits / nw);
  const int cu1 = (int)((long long)(c.cta() + 1) * kConsWarps * nunits / nw);
  const int r0 = cu0 / ub;
  const int nrk = cu1 > cu0 ? (cu1 - 1) / ub - r0 + 1 : 0;
  const int st0 = nrk > 0 ? m->ex_start[r0] : 0;
  const int ne0 = nrk > 0 ? m->ex_start[r0 + 1] - st0 : 0;
  const int st1 = nrk > 1 ? m->ex_start[r0 + 1] : 0;
  const int ne1 = nrk > 1 ? m->ex_start[r0 + 2] - st1 : 0;
  for (int q = c.tid(); q < I / 8; q += kConsThreads)
    *reinterpret_cast<uint4*>(Ag + a_chunk_off(32, q, I)) = make_uint4(0, 0, 0, 0);
  {
    const int per = I / 16, nitems = (ne0 + ne1) * per;
    if (nitems == 0)
      for (int j = pre; j < kXStages - 1 && j < nsteps; ++j) issue_step(j);
    for (int base = 0; base < nitems; base += 8 * kConsThreads) {
      uint2 cw[8];
      uint32_t sb[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int q = base + k * kConsThreads + c.tid();
        if (q < nitems) {
          const int i = q / per, blk = q % per;
          const int slot = i < ne0 ? m->ex_slots[st0 + i] : m->ex_slots[st1 + i - ne0];
          cw[k] = __ldcg(reinterpret_cast<const uint2*>(a.s.sq_codes + (size_t)slot * (I / 2) + blk * 8));
          sb[k] = __ldcg(a.s.sq_scales + (size_t)slot * (I / 16) + blk);
        }
      }
      if (base == 0) {
        stamp(c, 35);
        // any first steps not yet in flight, behind the intermediates' loads
        for (int j = pre; j < kXStages - 1 && j < nsteps; ++j) issue_step(j);
        stamp(c, 39);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int q = base + k * kConsThreads + c.tid();
        if (q < nitems) {
          const int i = q / per, blk = q % per;
          const int row = i < ne0 ? i : 16 + (i - ne0);
          const uint32_t scf = e4m3x2_to_f16x2(sb[k] | (sb[k] << 8));
          uint32_t out[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) out[j] = hmul2(e2m1_byte_to_f16x2(j < 4 ? cw[k].x : cw[k].y, j & 3), scf);
          *reinterpret_cast<uint4*>(Ag + a_chunk_off(row, 2 * blk, I)) = make_uint4(out[0], out[1], out[2], out[3]);
          *reinterpret_cast<uint4*>(Ag + a_chunk_off(row, 2 * blk + 1, I)) =
              make_uint4(out[4], out[5], out[6], out[7]);
        }
      }
    }
  }
  stamp(c, 43);
  named_bar(1, kConsThreads);
  stamp(c, kSlotExpert + 3);

  const int g = c.lane() >> 2, cq = c.lane() & 3;
  float acc[2][4];
  int prow = 32, b = 0, st = 0, ne = 0;
  float tsd = 0.f;
#pragma unroll 1
  for (int j = 0; j < nsteps; ++j) {
    const int kc0 = 4 * (j % spu);
    if (kc0 == 0) {
      const int u = u0 + j / spu;
      const int rank = u / ub;
      b = u % ub;
      st = m->ex_start[rank];
      ne = m->ex_start[rank + 1] - st;
      const int fi = c.lane() & 15;
      prow = fi < ne ? (rank == r0 ? fi : 16 + fi) : 32;
      tsd = __ldg(a.cur.ts + 3 * m->used[rank] + 2);
#pragma unroll
      for (int x = 0; x < 2; ++x) acc[x][0] = acc[x][1] = acc[x][2] = acc[x][3] = 0.f;
      if (j > 0) g2_prefetch_unit(c, s2, u + 2 * kUnitsAhead, pol);
    }
    if (j + kXStages - 1 < nsteps) issue_step(j + kXStages - 1);
    if (!xstage_wait(c)) break;
    const uint32_t stage = c.xstage(c.xs_done);
#pragma unroll 1
    for (int h = 0; h < 4; ++h)
      if (kc0 + h < nkc) {
        uint32_t af[8][4];
        load_a_chunk(af, A, prow, I, kc0 + h, c.lane());
        fp4_block_mma(acc[0], af, stage + (2 * h) * kBlk4, c.lane());
        fp4_block_mma(acc[1], af, stage + (2 * h + 1) * kBlk4, c.lane());
      }
    __syncwarp();
    c.xs_done++;
    if (kc0 + 4 >= nkc) {
      // y rows of the unit's slots: acc[gr] rows 8 gr + {2c, 2c+1}; [0,1] slot g, [2,3] slot g+8
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int fi2 = g + 8 * hh;
        if (fi2 < ne) {
          const int slot = m->ex_slots[st + fi2];
          uint16_t* yr = a.s.y + (size_t)slot * P + 16 * b;
          st32(yr + 2 * cq, pack_bf16x2(acc[0][2 * hh] * tsd, acc[0][2 * hh + 1] * tsd));
          st32(yr + 8 + 2 * cq, pack_bf16x2(acc[1][2 * hh] * tsd, acc[1][2 * hh + 1] * tsd));
        }
      }
      // count the unit in for each of its tokens; the token's k-th arrival
      // at this 16-row block combines its k expert outputs there
      __threadfence();
      __syncwarp();
      bool last = false;
      int t_mine = 0;
      if (c.lane() < ne) {
        t_mine = m->ex_slots[st + c.lane()] / d.topk;
        uint32_t* cnt = a.s.mc_cnt + (size_t)t_mine * ub + b;
        last = atom_add_acqrel_gpu(cnt, 1u) == (uint32_t)(d.topk - 1);
        if (last) *cnt = 0u;  // every arrival of this launch is in: rearm
      }
      const unsigned done = __ballot_sync(0xffffffffu, last);
      if (done) {
        __threadfence();
        // completed tokens four at a time: lane 8 k + i combines output
        // pair i of the k-th one, all k expert outputs loaded up front
        const int ncomp = __popc(done);
        for (int base = 0; base < ncomp; base += 4) {
          const int k = base + (c.lane() >> 3), pi = c.lane() & 7;
          const int src = k < ncomp ? (int)__fns(done, 0, k + 1) : 0;
          const int t = __shfl_sync(0xffffffffu, t_mine, src);
          if (k < ncomp) {
            const int p = 16 * b + 2 * pi;
            uint32_t yv[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
              if (r < d.topk) yv[r] = ldcg32(a.s.y + (size_t)(t * d.topk + r) * P + p);
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int r = 0; r < 8; ++r)
              if (r < d.topk) {
                const float gt = m->topk_gate[t][r];
                s0 = fmaf(gt, bf16_lo(yv[r]), s0);
                s1 = fmaf(gt, bf16_hi(yv[r]), s1);
              }
            st32(a.s.mvec + (size_t)t * P + p, pack_bf16x2(s0, s1));
          }
        }
      }
    }
    if (j == 0) stamp(c, kSlotExpert + 4);
  }
  xstage_drain(c);
  stamp(c, kSlotExpert + 5);
  cin = c;
}

}  // namespace msk
