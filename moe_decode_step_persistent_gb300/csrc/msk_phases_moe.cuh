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

static_assert(kMaxT * 8 <= kConsThreads, "a compute thread places at most one slot");
static_assert(kMaxT == 2 * kConsWarps, "a warp ranks tokens w and w + 8");
static_assert(kMaxT <= 32, "token sets of an expert are 32-bit masks");

// Ranking key of candidate expert e with fp32 logit bits b: order-preserving
// logit bits above, 0xFFFF - e below, so the larger key is the larger logit
// and ties go to the smaller expert index; 0 = no candidate.
__device__ __forceinline__ uint64_t topk_key(uint32_t b, int e) {
  const uint32_t ob = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)ob << 32) | (uint32_t)(0xFFFF - e);
}
__device__ __forceinline__ uint64_t max_u64(uint64_t x, uint64_t y) { return x > y ? x : y; }

// Warp-wide largest 64-bit key: the largest upper half, then the largest
// lower half among the lanes that hold it (two warp reductions).
__device__ __forceinline__ uint64_t warp_max_key(uint64_t k) {
  const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(k >> 32));
  const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(k >> 32) == hi ? (uint32_t)k : 0u);
  return ((uint64_t)hi << 32) | lo;
}

static __device__ __noinline__ void topk_dispatch(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  Misc* m = c.misc();
  // GEMM1's activations (Q4(pooled) as f16, written in the router phase)
  // stream into the staging area meanwhile (gemm1_phase waits for them)
  stage_issue(c, a.s.a4, d.P);
  // warp w ranks tokens w and w + 8 side by side (two independent chains):
  // lane l holds the keys of experts l + 32 j and its best one.  A round
  // finds the warp's best key, the lane holding it retires it and takes its
  // next best; after round r, lane r holds the r-th choice.
  // all 16 loads in flight at once: unconditional, at clamped indices (in
  // bounds for any T, E), the candidates outside [T][E] masked afterwards
  uint32_t raw[2][8];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float* row = a.s.logits + (size_t)min(c.warp() + kConsWarps * i, d.T - 1) * d.E;
#pragma unroll
    for (int j = 0; j < 8; ++j) raw[i][j] = __float_as_uint(__ldcg(row + min(c.lane() + 32 * j, d.E - 1)));
  }
  uint64_t key[2][8], lb[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = c.warp() + kConsWarps * i;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = c.lane() + 32 * j;
      key[i][j] = (t < d.T && e < d.E) ? topk_key(raw[i][j], e) : 0ull;
    }
  }
  stamp(c, 30);
#pragma unroll
  for (int i = 0; i < 2; ++i)
    lb[i] = max_u64(max_u64(max_u64(key[i][0], key[i][1]), max_u64(key[i][2], key[i][3])),
                    max_u64(max_u64(key[i][4], key[i][5]), max_u64(key[i][6], key[i][7])));
  uint64_t mine[2] = {0ull, 0ull};
#pragma unroll 1
  for (int r = 0; r < d.topk; ++r) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint64_t best = warp_max_key(lb[i]);
      if (c.lane() == r) mine[i] = best;
      // keys are unique (the expert index is part of the key): only the
      // holder's keys change
#pragma unroll
      for (int j = 0; j < 8; ++j) key[i][j] = key[i][j] == best ? 0ull : key[i][j];
      lb[i] = max_u64(max_u64(max_u64(key[i][0], key[i][1]), max_u64(key[i][2], key[i][3])),
                      max_u64(max_u64(key[i][4], key[i][5]), max_u64(key[i][6], key[i][7])));
    }
  }
  stamp(c, 31);
  // softmax over the selected logits: lane r's exp, summed in rank order
  // (lanes top_k .. 7 add exact zeros)
#pragma unroll 1
  for (int i = 0; i < 2; ++i) {
    const int t = c.warp() + kConsWarps * i;
    const uint64_t mk = i ? mine[1] : mine[0];
    const uint32_t mob = (uint32_t)(mk >> 32);
    const float my_v = mk == 0 ? -CUDART_INF_F : __uint_as_float((mob & 0x80000000u) ? (mob & 0x7FFFFFFFu) : ~mob);
    const int my_e = mk == 0 ? 0 : 0xFFFF - (int)(mk & 0xFFFFu);
    const float top = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = c.lane() < d.topk ? expf(my_v - top) : 0.f;
    float sum = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) sum += __shfl_sync(0xffffffffu, ex, r);
    if (t < d.T && c.lane() < d.topk) {
      const int sl = t * d.topk + c.lane();
      m->slot_e[sl] = my_e;
      m->slot_gate[sl] = ex / sum;
      m->slot_tok[sl] = (uint8_t)t;
      atomicOr(&m->tok_mask[my_e], 1u << t);  // (zeroed at launch start)
    }
  }
  named_bar(1, kConsThreads);
  stamp(c, 14);  // top-k chosen (timing builds only: stamp is a no-op without a timeline)
  if (c.cta() == 0 && a.routing_out != nullptr)
    for (int i = c.tid(); i < d.T * d.topk; i += kConsThreads) a.routing_out[i] = m->slot_e[i];
  if (c.warp() == 0) {
    // lane l owns experts [8l, 8l + 8): used-expert ranks and slot offsets
    // by one warp scan of (experts used, slots) packed into one word
    int cnt[8], nu = 0, ns = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      cnt[j] = __popc(m->tok_mask[8 * c.lane() + j]);
      nu += cnt[j] > 0;
      ns += cnt[j];
    }
    const int own = (nu << 16) | ns;
    int incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (c.lane() >= o) incl += v;
    }
    int rank = (incl - own) >> 16, start = (incl - own) & 0xFFFF;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 8 * c.lane() + j;
      m->ex_first[e] = start;
      if (cnt[j] > 0) {
        m->used[rank] = e;
        m->ex_start[rank] = start;
        rank++;
        start += cnt[j];
      }
    }
    if (c.lane() == 31) {
      m->n_used = incl >> 16;
      m->ex_start[incl >> 16] = incl & 0xFFFF;
    }
  }
  named_bar(1, kConsThreads);
  // slots grouped by expert, ascending slot order inside a group (the slots
  // of one expert belong to distinct tokens: slot order is token order)
  if (c.tid() < d.T * d.topk) {
    const int s = c.tid(), e = m->slot_e[s], t = m->slot_tok[s];
    m->ex_slots[m->ex_first[e] + __popc(m->tok_mask[e] & ((1u << t) - 1u))] = (uint8_t)s;
  }
  named_bar(1, kConsThreads);
  stamp(c, 15);  // dispatch lists ready
}

// ---------------------------------------------------------------------------
// NVFP4 helpers
// ---------------------------------------------------------------------------

// acc += W (one 16-row x k128 NVFP4 tile in shared memory, the mma A
// operand) times X^T (eight tokens, f16 B fragments `bf` of the chunk's
// eight k16 steps); with `two`, also acc2 += W X2^T for tokens 8..15.  The
// tile is dequantised on the fly (E2M1 x E4M3 is exact in fp16): the lane's
// 16 scales (rows g and g + 8) are converted pairwise once, each k16 step
// takes them as broadcast halves, and code bytes go straight into the cvt.
// acc: {D[g][2c], D[g][2c+1], D[g+8][2c], D[g+8][2c+1]} (row, token).
__device__ __forceinline__ void fp4_tile_mma(float (&acc)[4], float (&acc2)[4], const uint32_t (&bf)[8][2],
                                             const uint32_t (&bf2)[8][2], bool two, uint32_t tile, int lane) {
  const uint4 c0 = lds128(tile + lane * 16), c1 = lds128(tile + 512 + lane * 16);
  const int g = lane >> 2;
  const uint2 sg = lds64(tile + 1024 + g * 8), sg8 = lds64(tile + 1024 + (g + 8) * 8);
  const uint32_t spg[4] = {e4m3_pair_to_f16x2(sg.x, 0), e4m3_pair_to_f16x2(sg.x, 1), e4m3_pair_to_f16x2(sg.y, 0),
                           e4m3_pair_to_f16x2(sg.y, 1)};
  const uint32_t spg8[4] = {e4m3_pair_to_f16x2(sg8.x, 0), e4m3_pair_to_f16x2(sg8.x, 1),
                            e4m3_pair_to_f16x2(sg8.y, 0), e4m3_pair_to_f16x2(sg8.y, 1)};
  const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t scg = f16x2_bcast(spg[s >> 1], s & 1), scg8 = f16x2_bcast(spg8[s >> 1], s & 1);
    uint32_t a[4];
    a[0] = hmul2(e2m1_byte_to_f16x2(cw[s], 0), scg);   // row g,     k 2c
    a[1] = hmul2(e2m1_byte_to_f16x2(cw[s], 1), scg8);  // row g + 8, k 2c
    a[2] = hmul2(e2m1_byte_to_f16x2(cw[s], 2), scg);   // row g,     k 2c + 8
    a[3] = hmul2(e2m1_byte_to_f16x2(cw[s], 3), scg8);  // row g + 8, k 2c + 8
    mma_f16(acc, a, bf[s][0], bf[s][1]);
    if (two) mma_f16(acc2, a, bf2[s][0], bf2[s][1]);
  }
}

// B fragments (eight k16 steps of a k128 chunk) for eight tokens from a
// gathered [rows][K] f16 matrix in the staging area: lane l addresses
// physical row prow (the row of token l % 8) for the 8x8 matrix l / 8.
__device__ __forceinline__ void load_b_chunk(uint32_t (&bf)[8][2], uint32_t A, int prow, int K, int kc, int lane) {
  const uint32_t rb_ = A + prow * a_row_bytes(K);
#pragma unroll
  for (int s2 = 0; s2 < 4; ++s2) {
    const int ch = ((kc * 128 + 32 * s2) >> 3) + (lane >> 3);
    uint32_t r[4];
    ldmatrix_x4(r, rb_ + (ch << 4));
    bf[2 * s2][0] = r[0];
    bf[2 * s2][1] = r[1];
    bf[2 * s2 + 1][0] = r[2];
    bf[2 * s2 + 1][1] = r[3];
  }
}

// acc[nt][i] with nt and i known only at run time, by selects (no local
// memory, one copy of the caller's code).
__device__ __forceinline__ float pick_acc(const float (&acc)[2][4], int nt, int i) {
  const float a0 = (i & 1) ? acc[0][1] : acc[0][0], a1 = (i & 1) ? acc[0][3] : acc[0][2];
  const float b0 = (i & 1) ? acc[1][1] : acc[1][0], b1 = (i & 1) ? acc[1][3] : acc[1][2];
  const float a = (i & 2) ? a1 : a0, bb = (i & 2) ? b1 : b0;
  return nt ? bb : a;
}

// Sixteen values of one token spread as two per lane over the eight lanes
// g = 0..7 of a column c (rows g and g + 8 of a 16-row tile): Q4 block
// scale (E4M3 of amax / 6, round-to-nearest-even) and the lane's two codes.
// All lanes take part (shuffles over lane bits 2..4).
struct Q4Col {
  uint32_t scale;
  float dec;
};
__device__ __forceinline__ Q4Col q4_col(float x0, float x1) {
  float amax = fmaxf(fabsf(x0), fabsf(x1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 8));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
  Q4Col r{0u, 0.f};
  if (amax == 0.f) return r;
  r.scale = f32_to_e4m3(amax / 6.0f);
  r.dec = e4m3_to_f32(r.scale);
  return r;
}


// The expert units of a GEMM are numbered row block major (unit u = block
// u / n_used of used expert u % n_used), so that every contiguous run holds
// the experts in the same proportion (experts with more than eight tokens
// cost more per unit).  The runs, one per compute warp of the grid, are
// owned outright (whole K): no cross-warp reduction is needed.
__device__ __forceinline__ void warp_run(int nunits, const Ctx& c, int& u0, int& u1) {
  // (warps x units < 2^32: at most 1,216 x 32,768)
  const uint32_t nw = (uint32_t)c.nctas() * kConsWarps, gw = (uint32_t)c.cta() * kConsWarps + c.warp();
  u0 = (int)(gw * (uint32_t)nunits / nw);
  u1 = (int)((gw + 1) * (uint32_t)nunits / nw);
}

// A warp's stream of expert weight units in steps of two k128 chunks (one
// contiguous range per step).  Unit u is block u / nu of used expert u % nu;
// cursors walk it without divisions.
struct XStream {
  const uint8_t* base;  // the layer's experts + the GEMM's region offset
  size_t eb;            // bytes per expert
  int ubytes, nu, nkc, u0, u1, nsteps;
};

struct XCursor {
  int rank, blk, kc0;
  __device__ void init(const XStream& s, int u) {
    rank = u % s.nu;
    blk = u / s.nu;
    kc0 = 0;
  }
  __device__ void next_unit(const XStream& s) {
    kc0 = 0;
    if (++rank == s.nu) {
      rank = 0;
      ++blk;
    }
  }
  __device__ void next_step(const XStream& s) {
    kc0 += 2;
    if (kc0 >= s.nkc) next_unit(s);
  }
  __device__ const uint8_t* unit(const XStream& s, const Misc* m) const {
    return s.base + (size_t)m->used[rank] * s.eb + (size_t)blk * s.ubytes;
  }
};

__device__ __forceinline__ XStream x_stream(const Ctx& c, bool g2) {
  const Dims& d = c.a()->dm;
  XStream s;
  s.nu = c.misc()->n_used;
  s.eb = expert_bytes(d.P, d.I);
  s.base = c.a()->cur.experts + (g2 ? expert_g1_bytes(d.P, d.I) : 0);
  s.ubytes = g2 ? g2_unit_bytes(d.I) : g1_unit_bytes(d.P);
  s.nkc = (g2 ? d.I : d.P) / 128;
  warp_run(s.nu * (g2 ? d.P / kG2Rows : d.I / kG1Rows), c, s.u0, s.u1);
  s.nsteps = (s.u1 - s.u0) * ((s.nkc + 1) / 2);
  return s;
}

// Issues the step at `cur` into this warp's next stage and advances `cur`.
__device__ __forceinline__ void x_issue(Ctx& c, const XStream& s, XCursor& cur, uint64_t pol) {
  if (c.lane() == 0) {
    const int nb = min(2, s.nkc - cur.kc0);
    const uint32_t bar = c.xbar(c.xs_issued);
    mbar_arrive_expect_tx(bar, 2 * nb * kTile4);
    bulk_g2s_hint(c.xstage(c.xs_issued), cur.unit(s, c.misc()) + (size_t)2 * cur.kc0 * kTile4, 2 * nb * kTile4, bar,
                  pol);
  }
  c.xs_issued++;
  cur.next_step(s);
}


// ---------------------------------------------------------------------------
// Q4 of the pooled activations, once per launch: each block quantises its
// share of the (token, 16-block) items from the pooled rows it has staged
// for the router and writes the dequantised f16 values for every block's
// GEMM1.  Eight threads share an item (two elements each; the block amax
// is folded over the eight).
// ---------------------------------------------------------------------------

static __device__ __noinline__ void quantize_pooled(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  const int P = d.P, per = P / 16, n = d.T * per;
  const uint8_t* Ag = c.smem() + kOffA;
  const int i0 = (int)((long long)c.cta() * n / c.nctas()), i1 = (int)((long long)(c.cta() + 1) * n / c.nctas());
  const int j = c.lane() & 7;  // this thread's element pair within the item
  // the loop condition is uniform per warp (the shuffles need every lane);
  // lane group lane / 8 takes item qb + lane / 8
  for (int qb = i0 + 4 * c.warp(); qb < i1; qb += kConsThreads / 8) {
    const int q = qb + (c.lane() >> 3);
    const bool live = q < i1;
    const int t = live ? q / per : 0, blk = live ? q % per : 0;
    uint32_t w = 0;
    if (live) w = *reinterpret_cast<const uint32_t*>(Ag + a_chunk_off(t, 2 * blk + (j >> 2), P) + 4 * (j & 3));
    const float x0 = bf16_lo(w), x1 = bf16_hi(w);
    float amax = fmaxf(fabsf(x0), fabsf(x1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    uint32_t out = 0;
    if (amax > 0.f) {
      const uint32_t sc = f32_to_e4m3(amax / 6.0f);
      const float dec = e4m3_to_f32(sc);
      if (dec > 0.f) out = hmul2(e2m1x2_to_f16x2(f32x2_to_e2m1x2(x0 / dec, x1 / dec)), e4m3x2_to_f16x2(sc | (sc << 8)));
    }
    if (live) *reinterpret_cast<uint32_t*>(a.s.a4 + (size_t)t * P + 16 * blk + 2 * j) = out;
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
  const uint64_t pol = policy_evict_first();
  const XStream xs = x_stream(c, false);
  const int nkc = xs.nkc, nsteps = xs.nsteps;
  XCursor ic;  // issue and compute cursors
  ic.init(xs, xs.u0);
  XCursor cc = ic;
  // x = Q4(pooled) dequantised (f16 [17][P], row 16 = zeros): its copies
  // were issued during the top-k
  for (int q = c.tid(); q < P / 8; q += kConsThreads)
    *reinterpret_cast<uint4*>(Ag + a_chunk_off(16, q, P)) = make_uint4(0, 0, 0, 0);
  // the warp's first steps: in flight while the activations land
  for (int j = 0; j < kXStages - 1 && j < nsteps; ++j) x_issue(c, xs, ic, pol);
  stage_wait(c);
  named_bar(1, kConsThreads);
  stamp(c, kSlotExpert + 0);

  const int g = c.lane() >> 2, cq = c.lane() & 3;
  // acc[gu][nt]: gate / up, tokens 0..7 / 8..15 of the unit's expert
  float acc[2][2][4];
  int prow = 16, prow2 = 16, b = 0, st = 0, ne = 0;
  bool two = false;
  float tsg = 0.f, tsu = 0.f;
#pragma unroll 1
  for (int j = 0; j < nsteps; ++j) {
    const int kc0 = cc.kc0;
    if (kc0 == 0) {
      const int rank = cc.rank;
      const int e = m->used[rank];
      b = cc.blk;
      st = m->ex_start[rank];
      ne = m->ex_start[rank + 1] - st;
      two = ne > 8;
      const int r8 = c.lane() & 7;
      prow = r8 < ne ? m->slot_tok[m->ex_slots[st + r8]] : 16;
      prow2 = r8 + 8 < ne ? m->slot_tok[m->ex_slots[st + r8 + 8]] : 16;
      tsg = __ldg(a.cur.ts + 3 * e);
      tsu = __ldg(a.cur.ts + 3 * e + 1);
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 2; ++y) acc[x][y][0] = acc[x][y][1] = acc[x][y][2] = acc[x][y][3] = 0.f;
    }
    if (j + kXStages - 1 < nsteps) x_issue(c, xs, ic, pol);
    if (!xstage_wait(c)) break;
    const uint32_t stage = c.xstage(c.xs_done);
#pragma unroll 1
    for (int h = 0; h < 2; ++h)
      if (kc0 + h < nkc) {
        uint32_t bf[8][2], bf2[8][2];
        load_b_chunk(bf, A, prow, P, kc0 + h, c.lane());
        if (two) load_b_chunk(bf2, A, prow2, P, kc0 + h, c.lane());
        fp4_tile_mma(acc[0][0], acc[0][1], bf, bf2, two, stage + (2 * h) * kTile4, c.lane());
        fp4_tile_mma(acc[1][0], acc[1][1], bf, bf2, two, stage + (2 * h + 1) * kTile4, c.lane());
      }
    __syncwarp();
    c.xs_done++;
    if (kc0 + 2 >= nkc) {
      // SwiGLU of this unit's 16 rows (lane: rows g, g + 8; tokens 2c, 2c + 1
      // of each eight), then Q4 per (token, 16 rows): the 16 values of a
      // token sit in the eight lanes of its column; an even-g lane packs
      // rows (g, g + 1) and (g + 8, g + 9) with its neighbour's values.
      // One pass per token column q = (eight-token tile, parity): a loop
      // with the accumulators picked by selects keeps one copy of the code.
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        const int nt = q >> 1, ev = q & 1;
        if (nt == 1 && !two) break;  // (uniform over the warp)
        const int tok = 8 * nt + 2 * cq + ev;  // token index within the expert's slots
        float sv[2];
#pragma unroll
        for (int r8 = 0; r8 < 2; ++r8) {
          const float gv = pick_acc(acc[0], nt, 2 * r8 + ev) * tsg, uv = pick_acc(acc[1], nt, 2 * r8 + ev) * tsu;
          sv[r8] = gv / (1.0f + expf(-gv)) * uv;
        }
        const Q4Col qc = q4_col(sv[0], sv[1]);
        const float o0 = __shfl_xor_sync(0xffffffffu, sv[0], 4);
        const float o1 = __shfl_xor_sync(0xffffffffu, sv[1], 4);
        if (tok < ne) {
          // codes in GEMM2's B-fragment order: the pair (k, k + 1) of chunk
          // kc, k16 step s, half k8, column c at byte 64 kc + 16 c + 2 s + k8
          const int slot = m->ex_slots[st + tok];
          uint8_t* codes = a.s.sq_codes + (size_t)slot * (d.I / 2) + 64 * (b >> 3) + 8 * g + 2 * (b & 7);
          if ((g & 1) == 0) {
            uint32_t lo = 0u, hi = 0u;
            if (qc.dec > 0.f) {
              lo = f32x2_to_e2m1x2(sv[0] / qc.dec, o0 / qc.dec);
              hi = f32x2_to_e2m1x2(sv[1] / qc.dec, o1 / qc.dec);
            }
            codes[0] = (uint8_t)lo;
            codes[1] = (uint8_t)hi;
          }
          if (g == 0) a.s.sq_scales[(size_t)slot * (d.I / 16) + b] = (uint8_t)qc.scale;
        }
      }
    }
    if (j == 0) stamp(c, kSlotExpert + 1);
    cc.next_step(xs);
  }
  xstage_drain(c);
  stamp(c, kSlotExpert + 2);
  if (!aborted(c)) {
    // head start for GEMM2 (its weights do not depend on GEMM1): this
    // warp's first steps stream in while the grid waits at the barrier
    const XStream x2 = x_stream(c, true);
    XCursor ic2;
    ic2.init(x2, x2.u0);
    for (int j = 0; j < kXStages - 1 && j < x2.nsteps; ++j) x_issue(c, x2, ic2, pol);
  }
  cin = c;
}

// ---------------------------------------------------------------------------
// expert GEMM2: unit = (expert, 16 output rows); y = rb(s_q W_down^T), then
// the gated combine m[t] = rb(sum_r gate[t][r] y[t k + r]) (rank order) by
// whichever unit completes a (token, 16-row block) last
// ---------------------------------------------------------------------------

// GEMM2's B operand straight from the fp4 intermediates in global memory:
// lane (g, c) reads its slot's 16 code bytes of a k128 chunk (fragment
// order, written so by GEMM1) and the chunk's 8 block scales; slot < 0
// (no token) gives zeros.
struct B4 {
  uint4 c;
  uint2 s;
};

__device__ __forceinline__ B4 ld_b4(const LaunchArgs& a, int slot, int kc, int cq, int I) {
  B4 r;
  r.c = make_uint4(0, 0, 0, 0);
  r.s = make_uint2(0, 0);
  if (slot >= 0) {
    r.c = __ldcg(reinterpret_cast<const uint4*>(a.s.sq_codes + (size_t)slot * (I / 2) + 64 * kc + 16 * cq));
    r.s = __ldcg(reinterpret_cast<const uint2*>(a.s.sq_scales + (size_t)slot * (I / 16) + 8 * kc));
  }
  return r;
}

// Dequantised f16 B fragments of the chunk's eight k16 steps.
__device__ __forceinline__ void b4_frags(uint32_t (&bf)[8][2], const B4& b) {
  const uint32_t w[4] = {b.c.x, b.c.y, b.c.z, b.c.w};
  const uint32_t sp[4] = {e4m3_pair_to_f16x2(b.s.x, 0), e4m3_pair_to_f16x2(b.s.x, 1), e4m3_pair_to_f16x2(b.s.y, 0),
                          e4m3_pair_to_f16x2(b.s.y, 1)};
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t sc = f16x2_bcast(sp[s >> 1], s & 1);
    bf[s][0] = hmul2(e2m1_byte_to_f16x2(w[s >> 1], 2 * (s & 1)), sc);
    bf[s][1] = hmul2(e2m1_byte_to_f16x2(w[s >> 1], 2 * (s & 1) + 1), sc);
  }
}

static __device__ __noinline__ void gemm2_phase(Ctx& cin) {
  Ctx c = cin;  // register copy of the stage counters (written back at exit)
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  Misc* m = c.misc();
  const int I = d.I, P = d.P;
  const XStream xs = x_stream(c, true);
  const int nkc = xs.nkc, nsteps = xs.nsteps, ub = d.P / kG2Rows;
  const uint64_t pol = policy_evict_first();
  XCursor ic;  // issue, compute and B-operand cursors
  ic.init(xs, xs.u0);
  XCursor cc = ic, bc = ic;
  // steps already issued at the end of GEMM1
  const int pre = (int)(c.xs_issued - c.xs_done);
  for (int k = 0; k < pre; ++k) ic.next_step(xs);
  for (int j = pre; j < kXStages - 1 && j < nsteps; ++j) x_issue(c, xs, ic, pol);
  stamp(c, kSlotExpert + 3);

  const int g = c.lane() >> 2, cq = c.lane() & 3;
  // the B operand (fp4 intermediates of the unit's slots) of a step, one
  // step ahead: [chunk h][token tile nt]
  auto load_step_b = [&](B4 (&bb)[2][2]) {
    const int rank = bc.rank, kc0 = bc.kc0;
    bc.next_step(xs);
    const int st_ = m->ex_start[rank], ne_ = m->ex_start[rank + 1] - st_;
    const int s0 = g < ne_ ? m->ex_slots[st_ + g] : -1;
    const int s1 = g + 8 < ne_ ? m->ex_slots[st_ + g + 8] : -1;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const bool in = kc0 + h < nkc;
      bb[h][0] = ld_b4(a, in ? s0 : -1, kc0 + h, cq, I);
      bb[h][1] = ld_b4(a, in && ne_ > 8 ? s1 : -1, kc0 + h, cq, I);
    }
  };
  B4 bcur[2][2], bnxt[2][2];
  if (nsteps > 0) load_step_b(bcur);
  // acc[half][nt]: output rows 0..15 / 16..31 of the unit, tokens 0..7 / 8..15
  float acc[2][2][4];
  int b = 0, st = 0, ne = 0;
  bool two = false;
  float tsd = 0.f;
#pragma unroll 1
  for (int j = 0; j < nsteps; ++j) {
    const int kc0 = cc.kc0;
    if (kc0 == 0) {
      const int rank = cc.rank;
      b = cc.blk;
      st = m->ex_start[rank];
      ne = m->ex_start[rank + 1] - st;
      two = ne > 8;
      tsd = __ldg(a.cur.ts + 3 * m->used[rank] + 2);
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 2; ++y) acc[x][y][0] = acc[x][y][1] = acc[x][y][2] = acc[x][y][3] = 0.f;
    }
    if (j + kXStages - 1 < nsteps) x_issue(c, xs, ic, pol);
    if (j + 1 < nsteps) load_step_b(bnxt);
    if (!xstage_wait(c)) break;
    const uint32_t stage = c.xstage(c.xs_done);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (kc0 + h < nkc) {
        uint32_t bf[8][2], bf2[8][2];
        b4_frags(bf, bcur[h][0]);
        if (two) b4_frags(bf2, bcur[h][1]);
        fp4_tile_mma(acc[0][0], acc[0][1], bf, bf2, two, stage + (2 * h) * kTile4, c.lane());
        fp4_tile_mma(acc[1][0], acc[1][1], bf, bf2, two, stage + (2 * h + 1) * kTile4, c.lane());
      }
    __syncwarp();
    c.xs_done++;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      bcur[h][0] = bnxt[h][0];
      bcur[h][1] = bnxt[h][1];
    }
    if (kc0 + 2 >= nkc) {
      // y rows of the unit's slots: lane holds rows 16 half + g (+ 8) for
      // tokens 2c, 2c + 1 (of each eight); an even-g lane stores rows
      // (g, g + 1) and (g + 8, g + 9) as bf16 pairs with its neighbour's.
      // One pass per (half, token column); accumulators picked by selects.
#pragma unroll 1
      for (int q = 0; q < 8; ++q) {
        const int hf = q >> 2, nt = (q >> 1) & 1, ev = q & 1;
        if (nt == 1 && !two) continue;  // (uniform over the warp)
        const float v0 = (hf ? pick_acc(acc[1], nt, ev) : pick_acc(acc[0], nt, ev)) * tsd;
        const float v1 = (hf ? pick_acc(acc[1], nt, 2 + ev) : pick_acc(acc[0], nt, 2 + ev)) * tsd;
        const float o0 = __shfl_xor_sync(0xffffffffu, v0, 4), o1 = __shfl_xor_sync(0xffffffffu, v1, 4);
        const int tok = 8 * nt + 2 * cq + ev;
        if ((g & 1) == 0 && tok < ne) {
          const int slot = m->ex_slots[st + tok];
          uint16_t* yr = a.s.y + (size_t)slot * P + kG2Rows * b + 16 * hf;
          st32(yr + g, pack_bf16x2(v0, o0));
          st32(yr + 8 + g, pack_bf16x2(v1, o1));
        }
      }
      // count the unit in for each of its tokens; the token's k-th arrival
      // at this 32-row block combines its k expert outputs there
      __threadfence();
      __syncwarp();
      bool last = false;
      int t_mine = 0;
      if (c.lane() < ne) {
        t_mine = m->slot_tok[m->ex_slots[st + c.lane()]];
        uint32_t* cnt = a.s.mc_cnt + (size_t)t_mine * ub + b;
        last = atom_add_acqrel_gpu(cnt, 1u) == (uint32_t)(d.topk - 1);
        if (last) *cnt = 0u;  // every arrival of this launch is in: rearm
      }
      const unsigned done = __ballot_sync(0xffffffffu, last);
      if (done) {
        __threadfence();
        // completed tokens two at a time: lane 16 k + i combines output
        // pair i of the k-th one, all k expert outputs loaded up front
        const int ncomp = __popc(done);
        for (int base = 0; base < ncomp; base += 2) {
          const int k = base + (c.lane() >> 4), pi = c.lane() & 15;
          const int src = k < ncomp ? (int)__fns(done, 0, k + 1) : 0;
          const int t = __shfl_sync(0xffffffffu, t_mine, src);
          if (k < ncomp) {
            const int p = kG2Rows * b + 2 * pi;
            uint32_t yv[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
              if (r < d.topk) yv[r] = ldcg32(a.s.y + (size_t)(t * d.topk + r) * P + p);
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int r = 0; r < 8; ++r)
              if (r < d.topk) {
                const float gt = m->slot_gate[t * d.topk + r];
                s0 = fmaf(gt, bf16_lo(yv[r]), s0);
                s1 = fmaf(gt, bf16_hi(yv[r]), s1);
              }
            st32(a.s.mvec + (size_t)t * P + p, pack_bf16x2(s0, s1));
          }
        }
      }
    }
    if (j == 0) stamp(c, kSlotExpert + 4);
    cc.next_step(xs);
  }
  xstage_drain(c);
  stamp(c, kSlotExpert + 5);
  cin = c;
}

}  // namespace msk
