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

static __device__ void topk_dispatch(Ctx& c) {
  const LaunchArgs& a = *c.a;
  const Dims& d = a.dm;
  Misc* m = c.misc;
  for (int t = c.warp; t < d.T; t += kConsWarps) {
    float v[8];
    int taken = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = c.lane + 32 * j;
      v[j] = e < d.E ? __ldcg(a.s.logits + (size_t)t * d.E + e) : -CUDART_INF_F;
    }
    float sel_v[8];
    for (int r = 0; r < d.topk; ++r) {
      float bv = -CUDART_INF_F;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = c.lane + 32 * j;
        if (e < d.E && !((taken >> j) & 1) && (v[j] > bv || (v[j] == bv && e < be))) {
          bv = v[j];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == c.lane) taken |= 1 << (be >> 5);
      sel_v[r] = bv;
      if (c.lane == 0) m->topk_idx[t][r] = be;
    }
    if (c.lane == 0) {
      float s = 0.f;
      for (int r = 0; r < d.topk; ++r) s += expf(sel_v[r] - sel_v[0]);
      for (int r = 0; r < d.topk; ++r) m->topk_gate[t][r] = expf(sel_v[r] - sel_v[0]) / s;
    }
  }
  named_bar(1, kConsThreads);
  if (c.cta == 0 && a.routing_out != nullptr)
    for (int i = c.tid; i < d.T * d.topk; i += kConsThreads) a.routing_out[i] = m->topk_idx[i / d.topk][i % d.topk];
  if (c.warp == 0) {
    const int nslots = d.T * d.topk;
    for (int e = c.lane; e < 256; e += 32) m->ex_count[e] = 0;
    __syncwarp();
    for (int s = c.lane; s < nslots; s += 32) atomicAdd(&m->ex_count[m->topk_idx[s / d.topk][s % d.topk]], 1);
    __syncwarp();
    // lane l owns experts [8l, 8l + 8): ranks and slot offsets by warp scans
    int nu = 0, ns = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int cnt = m->ex_count[8 * c.lane + j];
      nu += cnt > 0;
      ns += cnt;
    }
    int nu_x = nu, ns_x = ns;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a1 = __shfl_up_sync(0xffffffffu, nu_x, o), a2 = __shfl_up_sync(0xffffffffu, ns_x, o);
      if (c.lane >= o) {
        nu_x += a1;
        ns_x += a2;
      }
    }
    int rank = nu_x - nu, start = ns_x - ns;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = 8 * c.lane + j;
      const int cnt = m->ex_count[e];
      if (cnt > 0) {
        m->used[rank] = e;
        m->ex_start[rank] = start;
        m->cursor[e] = start;
        rank++;
        start += cnt;
      }
    }
    if (c.lane == 31) {
      m->n_used = nu_x;
      m->ex_start[nu_x] = ns_x;
    }
    __syncwarp();
    // slots grouped by expert, ascending slot order inside a group
    for (int b0 = 0; b0 < nslots; b0 += 32) {
      const int s = b0 + c.lane;
      const int e = s < nslots ? m->topk_idx[s / d.topk][s % d.topk] : -1 - c.lane;
      const unsigned mask = __match_any_sync(0xffffffffu, e);
      const int rk = __popc(mask & ((1u << c.lane) - 1u));
      int base = 0;
      if (s < nslots) base = m->cursor[e];
      __syncwarp();
      if (s < nslots) {
        m->ex_slots[base + rk] = (uint8_t)s;
        if (rk == 0) m->cursor[e] = base + __popc(mask);
      }
      __syncwarp();
    }
    if (c.lane == 0) mbar_arrive(c.bar(BAR_DISPATCH));  // the producer may stream expert tiles
  }
  named_bar(1, kConsThreads);
}

// ---------------------------------------------------------------------------
// NVFP4 helpers
// ---------------------------------------------------------------------------

// One 8-row x k128 block against the 16-row A operand held in `af`:
// codes (this lane's 16 bytes) and scales (row g's 8 bytes) from shared.
__device__ __forceinline__ void fp4_block_mma(float (&acc)[4], const uint32_t (&af)[8][4], uint32_t blk,
                                              int lane) {
  const uint4 cw = lds128(blk + lane * 16);
  const uint2 sw = lds64(blk + 512 + (lane >> 2) * 8);
  const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t two = (cws[s >> 1] >> (16 * (s & 1))) & 0xFFFFu;
    const uint32_t sb = ((s < 4 ? sw.x : sw.y) >> (8 * (s & 3))) & 0xFFu;
    const uint32_t scf = e4m3x2_to_f16x2(sb | (sb << 8));
    const uint32_t b0 = hmul2(e2m1x2_to_f16x2(two & 0xFF), scf);
    const uint32_t b1 = hmul2(e2m1x2_to_f16x2(two >> 8), scf);
    mma_f16(acc, af[s], b0, b1);
  }
}

// A fragments (8 k16 steps of a k128 chunk) from a gathered [17][K] f16
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

// ---------------------------------------------------------------------------
// expert GEMM1 (+ SwiGLU + Q4): unit = (expert, 16 intermediate rows)
// ---------------------------------------------------------------------------

static __device__ void gemm1_phase(Ctx& c) {
  const LaunchArgs& a = *c.a;
  const Dims& d = a.dm;
  Misc* m = c.misc;
  const int P = d.P;
  uint8_t* Ag = c.smem + kOffA;
  const uint32_t A = c.sbase + kOffA;
  // a = Q4(pooled) dequantised, as f16 [17][P] (row 16 = zeros)
  for (int q = c.tid; q < kMaxT * (P / 16) + (P / 8); q += kConsThreads) {
    if (q >= kMaxT * (P / 16)) {
      *reinterpret_cast<uint4*>(Ag + a_chunk_off(16, q - kMaxT * (P / 16), P)) = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int t = q / (P / 16), blk = q % (P / 16);
    uint32_t out[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (t < d.T) {
      const uint4* src = reinterpret_cast<const uint4*>(a.s.pooled + (size_t)t * P + blk * 16);
      const uint4 v0 = __ldcg(src), v1 = __ldcg(src + 1);
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
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
    }
    *reinterpret_cast<uint4*>(Ag + a_chunk_off(t, 2 * blk, P)) = make_uint4(out[0], out[1], out[2], out[3]);
    *reinterpret_cast<uint4*>(Ag + a_chunk_off(t, 2 * blk + 1, P)) = make_uint4(out[4], out[5], out[6], out[7]);
  }
  named_bar(1, kConsThreads);
  const int red_off = kOffA + 17 * P * 2;
  float* red = reinterpret_cast<float*>(c.smem + red_off);  // [2][8][32][16]
  const ExpertSched sch = expert_sched(a, a.cur, m->n_used, true, c.cta, c.nctas);
  const int g = c.lane >> 2, cq = c.lane & 3;
  for (int ui = 0; ui < sch.nu; ++ui) {
    const int u = sch.u0 + ui;
    const int rank = u / sch.ublocks, b = u % sch.ublocks;
    const int e = m->used[rank];
    const int st = m->ex_start[rank], ne = m->ex_start[rank + 1] - st;
    const int fi = c.lane & 15;
    const int prow = fi < ne ? m->ex_slots[st + fi] / d.topk : 16;
    float acc[2][2][4];
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int y = 0; y < 2; ++y) acc[x][y][0] = acc[x][y][1] = acc[x][y][2] = acc[x][y][3] = 0.f;
    uint32_t af[8][4];
    for (int t = 0; t < sch.tpu; ++t) {
      const int kh = t >> 1, gu = t & 1;
      const int nk = min(8, sch.nkc - 8 * kh);
      const bool ok = wait_tile(c);
      if (ok && c.warp < nk) {
        const int kc = 8 * kh + c.warp;
        if (gu == 0) load_a_chunk(af, A, prow, P, kc, c.lane);
        const uint32_t slot = c.slot_addr(c.seq % kSlots);
#pragma unroll
        for (int gr = 0; gr < 2; ++gr) {
          const uint32_t blk = slot + (gr * nk + c.warp) * kBlk4;
          if (gu == 0) fp4_block_mma(acc[0][gr], af, blk, c.lane);
          else fp4_block_mma(acc[1][gr], af, blk, c.lane);
        }
      }
      release_tile(c);
    }
    float* rb_ = red + (ui & 1) * (kConsWarps * 32 * 16);
    float4* my = reinterpret_cast<float4*>(rb_ + (c.warp * 32 + c.lane) * 16);
    my[0] = make_float4(acc[0][0][0], acc[0][0][1], acc[0][0][2], acc[0][0][3]);
    my[1] = make_float4(acc[0][1][0], acc[0][1][1], acc[0][1][2], acc[0][1][3]);
    my[2] = make_float4(acc[1][0][0], acc[1][0][1], acc[1][0][2], acc[1][0][3]);
    my[3] = make_float4(acc[1][1][0], acc[1][1][1], acc[1][1][2], acc[1][1][3]);
    named_bar(1, kConsThreads);
    if (c.warp == (ui & (kConsWarps - 1))) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.f;
      for (int w = 0; w < kConsWarps; ++w) {
        const float4* p = reinterpret_cast<const float4*>(rb_ + (w * 32 + c.lane) * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 f = p[q];
          v[4 * q] += f.x;
          v[4 * q + 1] += f.y;
          v[4 * q + 2] += f.z;
          v[4 * q + 3] += f.w;
        }
      }
      // v[0..3] gate rows {2c,2c+1} (slot g, g+8), v[4..7] gate rows {8+2c, 9+2c},
      // v[8..11] up rows {2c,2c+1}, v[12..15] up rows {8+2c, 9+2c}
      const float tsg = __ldg(a.cur.ts + 3 * e), tsu = __ldg(a.cur.ts + 3 * e + 1);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float s[4];
        const int idx[4] = {2 * hh, 2 * hh + 1, 4 + 2 * hh, 4 + 2 * hh + 1};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float gv = v[idx[j]] * tsg, uv = v[8 + idx[j]] * tsu;
          s[j] = gv / (1.0f + expf(-gv)) * uv;
        }
        const Q4Out q = q4_quad(s);
        const int fi2 = g + 8 * hh;
        if (fi2 < ne && !aborted(c)) {
          const int slot = m->ex_slots[st + fi2];
          uint8_t* codes = a.s.sq_codes + (size_t)slot * (d.I / 2);
          codes[8 * b + cq] = (uint8_t)q.byte_lo;
          codes[8 * b + 4 + cq] = (uint8_t)q.byte_hi;
          if (cq == 0) a.s.sq_scales[(size_t)slot * (d.I / 16) + b] = (uint8_t)q.scale;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// expert GEMM2: unit = (expert, 16 output rows); y = rb(s_q W_down^T)
// ---------------------------------------------------------------------------

static __device__ void gemm2_phase(Ctx& c) {
  const LaunchArgs& a = *c.a;
  const Dims& d = a.dm;
  Misc* m = c.misc;
  const int I = d.I;
  uint8_t* Ag = c.smem + kOffA;
  const uint32_t A = c.sbase + kOffA;
  for (int q = c.tid; q < I / 8; q += kConsThreads)
    *reinterpret_cast<uint4*>(Ag + a_chunk_off(16, q, I)) = make_uint4(0, 0, 0, 0);
  const int red_off = kOffA + 17 * I * 2;
  float* red = reinterpret_cast<float*>(c.smem + red_off);  // [2][8][32][8]
  const ExpertSched sch = expert_sched(a, a.cur, m->n_used, false, c.cta, c.nctas);
  const int g = c.lane >> 2, cq = c.lane & 3;
  int cur_e = -1;
  for (int ui = 0; ui < sch.nu; ++ui) {
    const int u = sch.u0 + ui;
    const int rank = u / sch.ublocks, b = u % sch.ublocks;
    const int e = m->used[rank];
    const int st = m->ex_start[rank], ne = m->ex_start[rank + 1] - st;
    if (e != cur_e) {
      // this expert's fp4 intermediates, dequantised to f16 rows 0..ne-1
      named_bar(1, kConsThreads);
      for (int q = c.tid; q < ne * (I / 16); q += kConsThreads) {
        const int i = q / (I / 16), blk = q % (I / 16);
        const int slot = m->ex_slots[st + i];
        const uint2 cw = __ldcg(reinterpret_cast<const uint2*>(a.s.sq_codes + (size_t)slot * (I / 2) + blk * 8));
        const uint32_t sb = __ldcg(a.s.sq_scales + (size_t)slot * (I / 16) + blk);
        const uint32_t scf = e4m3x2_to_f16x2(sb | (sb << 8));
        uint32_t out[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t byte = ((j < 4 ? cw.x : cw.y) >> (8 * (j & 3))) & 0xFFu;
          out[j] = hmul2(e2m1x2_to_f16x2(byte), scf);
        }
        *reinterpret_cast<uint4*>(Ag + a_chunk_off(i, 2 * blk, I)) = make_uint4(out[0], out[1], out[2], out[3]);
        *reinterpret_cast<uint4*>(Ag + a_chunk_off(i, 2 * blk + 1, I)) = make_uint4(out[4], out[5], out[6], out[7]);
      }
      named_bar(1, kConsThreads);
      cur_e = e;
    }
    const int fi = c.lane & 15;
    const int prow = fi < ne ? fi : 16;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    uint32_t af[8][4];
    for (int t = 0; t < sch.tpu; ++t) {
      const int nk = min(8, sch.nkc - 8 * t);
      const bool ok = wait_tile(c);
      if (ok && c.warp < nk) {
        const int kc = 8 * t + c.warp;
        load_a_chunk(af, A, prow, I, kc, c.lane);
        const uint32_t slot = c.slot_addr(c.seq % kSlots);
        fp4_block_mma(acc[0], af, slot + (0 * nk + c.warp) * kBlk4, c.lane);
        fp4_block_mma(acc[1], af, slot + (1 * nk + c.warp) * kBlk4, c.lane);
      }
      release_tile(c);
    }
    float* rb_ = red + (ui & 1) * (kConsWarps * 32 * 8);
    float4* my = reinterpret_cast<float4*>(rb_ + (c.warp * 32 + c.lane) * 8);
    my[0] = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
    my[1] = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
    named_bar(1, kConsThreads);
    if (c.warp == (ui & (kConsWarps - 1))) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.f;
      for (int w = 0; w < kConsWarps; ++w) {
        const float4* p = reinterpret_cast<const float4*>(rb_ + (w * 32 + c.lane) * 8);
        const float4 f0 = p[0], f1 = p[1];
        v[0] += f0.x; v[1] += f0.y; v[2] += f0.z; v[3] += f0.w;
        v[4] += f1.x; v[5] += f1.y; v[6] += f1.z; v[7] += f1.w;
      }
      const float tsd = __ldg(a.cur.ts + 3 * e + 2);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int fi2 = g + 8 * hh;
        if (fi2 < ne && !aborted(c)) {
          const int slot = m->ex_slots[st + fi2];
          uint16_t* yr = a.s.y + (size_t)slot * d.P + 16 * b;
          st32(yr + 2 * cq, pack_bf16x2(v[2 * hh] * tsd, v[2 * hh + 1] * tsd));
          st32(yr + 8 + 2 * cq, pack_bf16x2(v[4 + 2 * hh] * tsd, v[4 + 2 * hh + 1] * tsd));
        }
      }
    }
  }
}

// m[t][p] = rb(sum_r gate[t][r] * y[t k + r][p]), rank order
static __device__ void mcomb_phase(Ctx& c) {
  const LaunchArgs& a = *c.a;
  const Dims& d = a.dm;
  const int half = d.P / 2;
  const int total = d.T * half;
  const int q0 = (int)((long long)c.cta * total / c.nctas), q1 = (int)((long long)(c.cta + 1) * total / c.nctas);
  for (int q = q0 + c.tid; q < q1; q += kConsThreads) {
    const int t = q / half, p = 2 * (q % half);
    float s0 = 0.f, s1 = 0.f;
    for (int r = 0; r < d.topk; ++r) {
      const float gt = c.misc->topk_gate[t][r];
      const uint32_t yv = ldcg32(a.s.y + (size_t)(t * d.topk + r) * d.P + p);
      s0 = fmaf(gt, bf16_lo(yv), s0);
      s1 = fmaf(gt, bf16_hi(yv), s1);
    }
    st32(a.s.mvec + (size_t)t * d.P + p, pack_bf16x2(s0, s1));
  }
}

}  // namespace msk
