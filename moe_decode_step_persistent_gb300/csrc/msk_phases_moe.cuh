// Compute-warp phases, part 2: router top-k and dispatch, the NVFP4 expert
// GEMMs on the fifth-generation tensor cores, and the gated combine of
// expert outputs.
//
// Expert numerics follow the pages: expert weights in NVFP4 ([newruntime]
// "What happened"), the first expert GEMM's output quantised to fp4 and the
// second's kept in bf16 ([orcarouter] "Dove si colloca il confine del
// kernel").  Both GEMM inputs are NVFP4 (W4A4): the tensor cores multiply
// E2M1 codes with their E4M3 block scales and accumulate in fp32; the
// per-matrix tensor scales are applied to the fp32 sums.
#pragma once

#include "msk_phases_dense.cuh"
#include "msk_tc.cuh"

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
// Q4 of the pooled activations, once per launch: each block quantises its
// share of the (token, 16-block) items from the pooled rows it has staged
// for the router and writes the E2M1 codes and E4M3 scales that every
// block's GEMM1 reads as its token operand.  Eight threads share an item
// (two elements each; the block amax is folded over the eight).
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
    uint32_t sc = 0, byte = 0;
    if (amax > 0.f) {
      sc = f32_to_e4m3(amax / 6.0f);
      const float dec = e4m3_to_f32(sc);
      if (dec > 0.f) byte = f32x2_to_e2m1x2(x0 / dec, x1 / dec);
      else sc = 0;
    }
    if (live) {
      a.s.x4_codes[(size_t)t * (P / 2) + 8 * blk + j] = (uint8_t)byte;
      if (j == 0) a.s.x4_scales[(size_t)t * per + blk] = (uint8_t)sc;
    }
  }
}

// ---------------------------------------------------------------------------
// Expert GEMMs on the tensor cores (tcgen05 kind::mxf4nvf4, block-scaled
// NVFP4 with E4M3 scales per 16 elements, fp32 accumulation in tensor
// memory).  Weight rows are the MMA's M = 128, the (at most 16) token slots
// of an expert its N = 16, so each streamed weight byte is used once.
//
// Work items are units (GEMM g, used expert rank r, row block b): a GEMM1
// unit is 128 tile rows (64 gate and 64 up rows) over K = P, a GEMM2 unit
// 128 output rows over K = I.  The blocks' producers claim items one at a
// time from one queue of the launch (claim_index, resolve_item): every GEMM1 unit,
// expert-major, then the GEMM2 units in the order in which the experts'
// GEMM1 parts completed (the last GEMM1 epilogue warp of an expert appends
// it to the ready list).  So the blocks finish together, and GEMM2 starts
// on an expert as soon as its GEMM1 parts are done.
// Roles during the GEMMs:
//   producer warp  claims the items, posts each to the block's item queue
//                  and streams its weight stages (codes + scale chunks of
//                  kUStageK each) into kXSlots shared-memory slots;
//   compute warps  stage each item's token operand (xb_stage; two buffers,
//                  the next item's staged while the current one runs);
//   MMA warps      (lane 0 of each of kMmaIssuers) each copy the token
//                  operand's scale chunks of their MMAs into tensor memory,
//                  then per stage their half of the weights' chunks, issue
//                  their half of the stage's MMAs into their own set of the
//                  unit's accumulator (kAccs accumulators in turn), commit
//                  the stage back to the producer and the accumulator to
//                  the epilogue;
//   compute warps  read the accumulator (warp w: lanes 32 (w % 4) ..
//                  32 (w % 4) + 31, token columns 8 (w / 4) .. 8 (w / 4) + 7,
//                  both issuers' sets added) and run the GEMM's epilogue,
//                  each warp on its own; compute thread 0 counts a GEMM1
//                  unit in for its expert once every warp's part is stored.
// Every wait is bounded; on expiry the waiter records the error and the
// launch winds down (the tensor memory is released only after every issued
// tcgen05 operation has completed).
// ---------------------------------------------------------------------------

// Token operand of expert rank r into B buffer j: row n is slot n of the
// expert (GEMM1: Q4 of the slot's token's pooled vector; GEMM2: the slot's
// fp4 intermediate), codes in the tensor-core layout, then one 512-byte
// scale chunk per MMA (row n at 16 n: the slot's four block scales of the
// MMA; everything else zero).  Rows past the expert's slots are zero.
// Every copy is an asynchronous 16- or 4-byte copy, left in flight; the
// caller waits for them and orders them before the tensor core's reads
// (proxy fence + barrier).  All compute threads.
static __device__ __noinline__ void xb_stage(Ctx& c, int g, int r, int j) {
  const LaunchArgs& a = *c.a();
  const Misc* m = c.misc();
  const int K = g ? a.dm.I : a.dm.P, kc = K / 32, nmma = K / 64;
  uint8_t* B = c.smem() + kOffXB + j * kXBBytes;
  uint8_t* Bsf = B + kUN * K / 2;
  const uint32_t Bs = smem_u32(B), Bsfs = smem_u32(Bsf);
  const int st = m->ex_start[r], ne = m->ex_start[r + 1] - st;
  static_assert(kConsThreads == 16 * kUN && kConsThreads == 8 * 32, "operand staging thread mapping");
  {  // codes: thread (n, q0) copies chunks q0, q0 + 16, ... of row n
    const int n = c.tid() >> 4;
    const uint8_t* src = nullptr;
    if (n < ne) {
      const int slot = m->ex_slots[st + n];
      src = g ? a.s.sq_codes + (size_t)slot * (K / 2) : a.s.x4_codes + (size_t)m->slot_tok[slot] * (K / 2);
    }
    for (int q = c.tid() & 15; q < kc; q += 16) {
      if (src != nullptr) cp_async16(Bs + umma_code_off(kUN, n, 32 * q), src + 16 * q);
      else *reinterpret_cast<uint4*>(B + umma_code_off(kUN, n, 32 * q)) = make_uint4(0, 0, 0, 0);
    }
  }
  {  // scale chunks: thread (n, kk0) writes row n of chunks kk0, kk0 + 8, ...
    const int n = c.tid() & 31;
    const uint8_t* src = nullptr;
    if (n < ne) {
      const int slot = m->ex_slots[st + n];
      src = g ? a.s.sq_scales + (size_t)slot * (K / 16) : a.s.x4_scales + (size_t)m->slot_tok[slot] * (K / 16);
    }
    for (int kk = c.tid() >> 5; kk < nmma; kk += 8) {
      uint8_t* row = Bsf + 512 * kk + 16 * n;
      if (src != nullptr) {
        cp_async4(Bsfs + 512 * kk + 16 * n, src + 4 * kk);
        *reinterpret_cast<uint32_t*>(row + 4) = 0u;
        *reinterpret_cast<uint2*>(row + 8) = make_uint2(0u, 0u);
      } else {
        *reinterpret_cast<uint4*>(row) = make_uint4(0, 0, 0, 0);
      }
    }
  }
}

// The MMAs of a stage with kst / 64 of them that issuer i takes: kk in
// [i kn / kMmaIssuers, (i + 1) kn / kMmaIssuers).
__device__ __forceinline__ int x_kk0(int kn, int i) { return i * kn / kMmaIssuers; }

// MMA thread i: the token operand's scale chunks of buffer j for its MMAs
// into tensor-memory region j.
__device__ __forceinline__ void xmma_sfb(const Ctx& c, int K, int j, int i) {
  const uint32_t tb = c.misc()->tmem;
  const int nst = (K + kUStageK - 1) / kUStageK;
  for (int s = 0; s < nst; ++s) {
    const int kn = ustage_k(K, s) / 64;
    for (int kk = x_kk0(kn, i); kk < x_kk0(kn, i + 1); ++kk) {
      const int jm = (kUStageK / 64) * s + kk;
      tc_cp_sf(tb + tmem_sfb(j, jm), umma_desc(c.sbase() + kOffXB + j * kXBBytes + kUN * K / 2 + 512 * jm, 128, 128));
    }
  }
}

// MMA thread i: its half of one unit (K long, token operand in buffer j)
// into its half of the next accumulator: per stage the weight scale chunks
// and MMAs of its share, the stage committed back to the producer (which
// refills the slot once every issuer has committed); then the accumulator
// committed to the epilogue warps.  Returns false if a wait ran out or the
// launch aborted.
static __device__ __noinline__ bool xmma_unit(Ctx& cin, int K, int j, int i) {
  Ctx c = cin;  // register copy of the counters (written back at exit)
  const uint32_t tb = c.misc()->tmem;
  const uint32_t idesc = idesc_mxf4nvf4(kUN);
  const uint32_t B = c.sbase() + kOffXB + (uint32_t)j * kXBBytes;
  const uint32_t acc = c.xunit % kAccs;
  const int nst = (K + kUStageK - 1) / kUStageK;
  bool ok = true;
  if (c.xunit >= (uint32_t)kAccs)
    ok = mbar_wait(c.bar(BAR_ACCE + acc), ((c.xunit / kAccs) - 1) & 1, c.deadline(), c.abort_ptr());
  if (!ok && !aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -11);
  tc_fence_after();
  for (int s = 0; s < nst && ok; ++s) {
    const uint32_t slot = c.xseq % kXSlots;
    ok = mbar_wait(c.bar(BAR_XFULL + slot), (c.xseq / kXSlots) & 1, c.deadline(), c.abort_ptr());
    if (!ok) {
      if (!aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -12);
      break;
    }
    tc_fence_after();
    const int kst = ustage_k(K, s), kn = kst / 64, k0 = x_kk0(kn, i);
    const uint32_t sa = c.xstage(c.xseq);
    for (int kk = k0; kk < x_kk0(kn, i + 1); ++kk) {
      const int jm = (kUStageK / 64) * s + kk;  // MMA index along K
      tc_cp_sf(tb + tmem_sfa(slot, kk), umma_desc(sa + 64 * kst + 512 * kk, 128, 128));
      mma_mxf4nvf4(tb + tmem_acc(i, acc), umma_desc(sa + 4096 * kk, 16 * kURows, 128),
                   umma_desc(B + 512 * jm, 16 * kUN, 128), idesc, tb + tmem_sfa(slot, kk), tb + tmem_sfb(j, jm),
                   s > 0 || kk > k0);
    }
    tc_commit(c.bar(BAR_XEMPTY + slot));  // (the producer refills the slot once every issuer's MMAs on it are done)
    c.xseq++;
  }
  if (ok) {
    tc_commit(c.bar(BAR_ACCF + acc));
    c.xunit++;
  }
  cin = c;
  return ok;
}

// Waits (one lane, bounded) for accumulator use c.xunit to be complete;
// false (uniformly over the warp) if the wait ran out or the launch aborted.
__device__ __forceinline__ bool xacc_wait(const Ctx& c) {
  bool got = true;
  if (c.lane() == 0)
    got = mbar_wait(c.bar(BAR_ACCF + c.xunit % kAccs), (c.xunit / kAccs) & 1, c.deadline(), c.abort_ptr());
  if (!__shfl_sync(0xffffffffu, (int)got, 0)) return false;
  tc_fence_after();
  return true;
}

// This warp's 32 rows of token columns 8 h .. 8 h + 7 of accumulator use
// c.xunit (the issuers' halves added in issuer order).
__device__ __forceinline__ void xacc_ld8(const Ctx& c, int h, float (&v)[8]) {
  const uint32_t base = tmem_lane_addr(c.misc()->tmem, 32 * (c.warp() & 3), 8 * h);
  const int acc = (int)(c.xunit % kAccs);
  tmem_ld8(base + tmem_acc(0, acc), v);
#pragma unroll
  for (int i = 1; i < kMmaIssuers; ++i) {
    float w[8];
    tmem_ld8(base + tmem_acc(i, acc), w);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] += w[e];
  }
}

// Hands accumulator use c.xunit back to the MMA thread.
__device__ __forceinline__ void xacc_release(Ctx& c) {
  tc_fence_before();
  __syncwarp();
  if (c.lane() == 0) mbar_arrive(c.bar(BAR_ACCE + c.xunit % kAccs));
  c.xunit++;
}

// GEMM1 epilogue, warp w (quadrant q = w % 4, token half h = w / 4): lanes
// i < 16 hold gate row 64 b + 16 q + i, lanes 16 + i the up row with the
// same index (the tiled layout interleaves them), for slots 8 h .. 8 h + 7
// of the expert.  SwiGLU s = silu(g) u lands on lanes 0..15; then lanes
// 16..31 take over slots 8 h + 4 .. 8 h + 7 of lane i - 16, so that every
// lane quantises four values.  Q4 of each slot's 16 values (one block of 16
// intermediate rows, one 16-lane half): E4M3 scale of amax / 6, E2M1 codes
// of s / scale (IEEE division: the code decision), written to the slot's
// fp4 intermediate (the GEMM2 input).  The warp that completes an expert's
// count appends it to the launch's GEMM2 ready list.
static __device__ __noinline__ void xepi_gemm1(Ctx& cin, int r, int b) {
  Ctx c = cin;
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  const Misc* m = c.misc();
  const int q = c.warp() & 3, h = c.warp() >> 2, lane = c.lane(), i = lane & 15, up = lane >> 4;
  const int e = m->used[r], st = m->ex_start[r], ne = m->ex_start[r + 1] - st;
  if (xacc_wait(c)) {
    if (8 * h < ne) {  // (uniform over the warp)
      const float ts = __ldg(a.cur.ts + 3 * e + up);  // gate (lanes 0..15) or up (16..31)
      const int row = 64 * b + 16 * q + i;            // intermediate row of lane i
      float v[8];
      xacc_ld8(c, h, v);
      float x[4], am[4];
      {
        float sv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float g = v[j] * ts;
          const float uv = __shfl_xor_sync(0xffffffffu, g, 16);
          sv[j] = __fdividef(g, 1.0f + __expf(-g)) * uv;  // (lanes 16..31: unused)
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float hi = __shfl_xor_sync(0xffffffffu, sv[4 + j], 16);  // lane i's slot 4 + j, on lane 16 + i
          x[j] = up ? hi : sv[j];
          am[j] = fabsf(x[j]);
        }
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1)
#pragma unroll
        for (int j = 0; j < 4; ++j) am[j] = fmaxf(am[j], __shfl_xor_sync(0xffffffffu, am[j], o));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t sc = 0, code = 0;
        if (am[j] > 0.f) {
          sc = f32_to_e4m3(am[j] / 6.0f);
          const float dec = e4m3_to_f32(sc);
          if (dec > 0.f) code = f32x2_to_e2m1x2(x[j] / dec, 0.f) & 0xFu;
          else sc = 0;
        }
        // eight codes per 32-bit word: lanes 0..7 and 8..15 of each half
        uint32_t w = code << (4 * (i & 7));
        w |= __shfl_xor_sync(0xffffffffu, w, 1);
        w |= __shfl_xor_sync(0xffffffffu, w, 2);
        w |= __shfl_xor_sync(0xffffffffu, w, 4);
        const int n = 8 * h + 4 * up + j;
        if (n < ne) {
          const int slot = m->ex_slots[st + n];
          if ((lane & 7) == 0)
            *reinterpret_cast<uint32_t*>(a.s.sq_codes + (size_t)slot * (d.I / 2) + row / 2) = w;
          if (i == 0) a.s.sq_scales[(size_t)slot * (d.I / 16) + row / 16] = (uint8_t)sc;
        }
      }
    }
    xacc_release(c);
  }
  cin = c;
}

// Counts a GEMM1 unit's epilogue in for its expert (`it`, or nothing when
// it < 0), after every compute warp's stores of it: a block barrier, then
// compute thread 0's release add of the eight warps' parts (the barrier
// orders the other warps' stores before it).  The block that completes the
// expert's count appends the expert to the launch's GEMM2 ready list
// (through the counter's release sequence every part's stores are visible
// before the entry).  One thread waits for the atomic's reply, the other
// warps go on.
static __device__ __noinline__ void x_count(Ctx& c, int it) {
  if (it < 0) return;
  named_bar(1, kConsThreads);
  if (c.tid() == 0) {
    const LaunchArgs& a = *c.a();
    const int r = item_r(it), e = c.misc()->used[r];
    const uint32_t total = (uint32_t)(kConsWarps * (a.dm.I / 64));
    if (atom_add_acqrel_gpu(a.s.x1_done + e, (uint32_t)kConsWarps) + (uint32_t)kConsWarps == total) {
      const uint32_t pos = atomicAdd(a.s.xq, 1u);
      st_release_gpu(a.s.xq + 2 + pos, (uint32_t)r + 1u);
    }
  }
}

// GEMM2 epilogue of one unit (rank r, row block b), warp w (quadrant
// q = w % 4, token half h = w / 4): lane i holds output row 128 b + 32 q + i
// of slots 8 h .. 8 h + 7 of the expert; y = rb(acc * tensor scale) per
// slot (the gated combine of a token's expert outputs is the next phase).
static __device__ __noinline__ void xepi_gemm2(Ctx& cin, int r, int b) {
  Ctx c = cin;
  const LaunchArgs& a = *c.a();
  const Misc* m = c.misc();
  const int q = c.warp() & 3, h = c.warp() >> 2, lane = c.lane(), P = a.dm.P;
  const int e = m->used[r], st = m->ex_start[r], ne = m->ex_start[r + 1] - st;
  if (xacc_wait(c)) {
    if (8 * h < ne) {  // (uniform over the warp)
      const float ts = __ldg(a.cur.ts + 3 * e + 2);
      const int row = kURows * b + 32 * q + lane;
      float v[8];
      xacc_ld8(c, h, v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (8 * h + j < ne)
          a.s.y[(size_t)m->ex_slots[st + 8 * h + j] * P + row] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j] * ts));
    }
    xacc_release(c);
  }
  cin = c;
}

// Gated combine of the expert outputs, m[t] = rb(sum_r gate_r y[t k + r])
// in rank order, over the whole grid: item (token, 32-row block), a warp
// per item and a lane per row, every slot's value loaded at once.
static __device__ __noinline__ void moe_combine_phase(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  const Misc* m = c.misc();
  // every block is done with the GEMM1 counters and the GEMM2 queue (before
  // the grid barrier that ended GEMM2): rearm them for the next launch
  if (c.cta() == 0) {
    for (int e = c.tid(); e < d.E; e += kConsThreads) a.s.x1_done[e] = 0u;
    for (int i = c.tid(); i < d.E + 2; i += kConsThreads) a.s.xq[i] = 0u;
  }
  const int P = d.P, nblk = P / 32, nitems = d.T * nblk;
  for (int it = c.cta() * kConsWarps + c.warp(); it < nitems; it += c.nctas() * kConsWarps) {
    const int t = it / nblk, row = 32 * (it - t * nblk) + c.lane();
    uint16_t yv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < d.topk) yv[k] = __ldcg(a.s.y + (size_t)(t * d.topk + k) * P + row);
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < d.topk) acc = fmaf(m->slot_gate[t * d.topk + k], __uint_as_float((uint32_t)yv[k] << 16), acc);
    a.s.mvec[(size_t)t * P + row] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
  }
}

// Thread 0: polls until the producer posts item k (true) or the
// accumulator of the block's oldest unread unit (c.xunit) completes (false),
// whichever comes first.  On abort or past the deadline it returns true: the
// bounded wait that follows reports it.
__device__ __forceinline__ bool xq_poll(const Ctx& c, uint32_t k) {
  const uint32_t qb = c.bar(BAR_QFULL + (k & 1)), qp = (k >> 1) & 1;
  const uint32_t ab = c.bar(BAR_ACCF + c.xunit % kAccs), ap = (c.xunit / kAccs) & 1;
  const uint64_t dl = c.deadline();
  uint32_t spins = 0;
  while (true) {
    if (mbar_test_wait(qb, qp)) return true;
    if (mbar_test_wait(ab, ap)) return false;
    if ((++spins & 63) == 0 && (aborted(c) || gtimer() > dl)) return true;
  }
}

// How xq_stage waits for the item: until it is posted; not at all (-3 if
// not posted yet); or until it is posted or the oldest pending accumulator
// is complete (-3 in the latter case).
constexpr int XQ_WAIT = 0, XQ_NOW = 1, XQ_OR_ACC = 2;

// The compute warps' side of the block's k-th expert item, first half: the
// item from the queue (thread 0, bounded; published through shared memory),
// then, once the MMAs of item k - 2 are done with buffer k % 2, the
// asynchronous copies of its token operand into that buffer (left in
// flight: xq_publish waits for them).  Returns the item, -1 when there is
// none (or the launch is winding down), or -3 when `mode` gave up on it
// (nothing done).
static __device__ __noinline__ int xq_stage(Ctx& c, uint32_t k, int mode) {
  const uint32_t q = k & 1;
  volatile int* bc = &c.misc()->xq_bcast[q];
  if (c.tid() == 0) {
    int it = -1;
    const int first = k == 0 ? first_expert_item(c) : -4;
    if (first != -4) {  // preassigned: no need to wait for the producer's post
      it = first;
      mbar_arrive(c.bar(BAR_QEMPTY + q));
    } else if (mode == XQ_NOW && !mbar_test_wait(c.bar(BAR_QFULL + q), (k >> 1) & 1)) {
      it = -3;
    } else if (mode == XQ_OR_ACC && !xq_poll(c, k)) {
      it = -3;
    } else if (mbar_wait(c.bar(BAR_QFULL + q), (k >> 1) & 1, c.deadline(), c.abort_ptr())) {
      it = *(volatile int*)&c.misc()->xq_unit[q];
      mbar_arrive(c.bar(BAR_QEMPTY + q));
      if (it >= 0 && k >= 2 &&
          !mbar_wait(c.bar(BAR_BFREE + q), ((k >> 1) - 1) & 1, c.deadline(), c.abort_ptr())) {
        if (!aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -13);
        it = -1;
      }
    } else if (!aborted(c)) {
      raise_error(c, ERR_TIMEOUT_RING, -14);
    }
    *bc = it;
  }
  named_bar(1, kConsThreads);
  const int it = *bc;
  if (it < 0) return it;
  tc_fence_after();  // (the buffer's previous MMAs completed: ordered before the new writes)
  xb_stage(c, item_g(it), item_r(it), (int)q);
  return it;
}

// Second half: the copies landed; the operand is ordered before the tensor
// cores' reads and item k may start.  A pending GEMM1 count (`cnt`, see
// x_count) is made while the copies land.
static __device__ __noinline__ void xq_publish(Ctx& c, uint32_t k, int cnt) {
  x_count(c, cnt);
  cp_async_wait_all();
  fence_proxy_async_shared();  // the operand writes before the tensor core reads them
  named_bar(1, kConsThreads);
  if (c.tid() == 0) mbar_arrive(c.bar(BAR_B2RDY + (k & 1)));
}

__device__ __forceinline__ void x_epilogue(Ctx& c, int it) {
  if (item_g(it) == 0) xepi_gemm1(c, item_r(it), item_b(it));
  else xepi_gemm2(c, item_r(it), item_b(it));
}

// The expert GEMMs, every compute thread of the block.  While the tensor
// cores run item k, the compute warps copy item k + 1's token operand and,
// while those copies land, run item k - 1's epilogue (the epilogue lags two
// items, so the next operand is ready before the tensor cores finish the
// current item).  Item k + 1 is never waited for alone while an epilogue is
// pending: the producer may be waiting for an expert's GEMM1 parts to
// complete, and a pending epilogue may be one of them.  So, when item k + 1
// is not posted yet once item k - 1's epilogue is done, the warps wait for
// whichever comes first: its post (then it is staged as usual, ahead of
// item k's epilogue) or item k's accumulator (then that epilogue runs
// first).  The next layer's KV prefetch is issued once the first operand is
// staged.
static __device__ __forceinline__ void expert_gemms(Ctx& c) {
  int cur = xq_stage(c, 0, XQ_WAIT);  // item k, staged
  if (cur >= 0) xq_publish(c, 0, -1);
  stamp(c, kSlotExpert);
  prefetch_next_kv(c);
  // (a GEMM1 epilogue's count is made before any wait that depends on the
  // producer, which may be waiting for that very count)
  auto g1 = [](int it) { return it >= 0 && item_g(it) == 0 ? it : -1; };
  int prev = -1;  // item k - 1, epilogue pending
  for (uint32_t k = 0; cur >= 0; ++k) {
    int nx = xq_stage(c, k + 1, XQ_NOW);
    int cnt = -1;  // the GEMM1 item whose epilogue is not counted in yet
    if (prev >= 0) {
      x_epilogue(c, prev);
      cnt = g1(prev);
    }
    if (nx == -3) {
      x_count(c, cnt);
      cnt = -1;
      nx = xq_stage(c, k + 1, XQ_OR_ACC);
    }
    if (nx == -3) {
      x_epilogue(c, cur);
      x_count(c, g1(cur));
      cur = -1;
      nx = xq_stage(c, k + 1, XQ_WAIT);
    }
    // (the count after the publish: its round trip then overlaps the wait
    // for item k's MMAs that staging item k + 2 begins with)
    if (nx >= 0) xq_publish(c, k + 1, -1);
    x_count(c, cnt);
    prev = cur;
    cur = nx;
  }
  if (prev >= 0) {
    x_epilogue(c, prev);
    x_count(c, g1(prev));
  }
  stamp(c, kSlotExpert + 5);
}

// MMA warp i's whole launch (lane 0): the block's expert items as the queue
// delivers them (each item's token scale chunks for its MMAs, its share of
// the stages, then a commit that frees the operand buffer once every issuer
// has committed); then one commit that tracks every tcgen05 operation it
// issued (the tensor memory is released after every issuer's).
static __device__ void mma_warp(Ctx& c, int i) {
  if (c.lane() == 0) {
    const Dims& d = c.a()->dm;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
      const uint32_t q = k & 1;
      ok = mbar_wait(c.bar(BAR_QFULL + q), (k >> 1) & 1, c.deadline(), c.abort_ptr());
      if (!ok) break;
      const int it = *(volatile int*)&c.misc()->xq_unit[q];
      mbar_arrive(c.bar(BAR_QEMPTY + q));
      if (it < 0) break;
      ok = mbar_wait(c.bar(BAR_B2RDY + q), (k >> 1) & 1, c.deadline(), c.abort_ptr());
      if (!ok) {
        if (!aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -10);
        break;
      }
      tc_fence_after();
      const int K = item_g(it) ? d.I : d.P;
      xmma_sfb(c, K, (int)q, i);
      ok = xmma_unit(c, K, (int)q, i);
      tc_commit(c.bar(BAR_BFREE + q));  // once this item's MMAs are done, buffer q may take item k + 2
    }
    if (!ok && !aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -6);
    tc_commit(c.bar(BAR_TCDONE));
  }
}

}  // namespace msk
