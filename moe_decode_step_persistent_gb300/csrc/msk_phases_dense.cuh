// Compute-warp phases, part 1: activation staging, the dense projection
// engine (tokens as the 16-row A operand, weight rows as 8-column B tiles
// streamed through the ring), its epilogues, RoPE, split-KV GQA attention
// and the split combine.
#pragma once

#include <math_constants.h>

#include "msk_kernel_core.cuh"

namespace msk {

// The staging area holds a [16][K] 16-bit matrix with rows padded by 16
// bytes, so that the 8 rows an ldmatrix phase touches (same column) fall in
// 8 different bank groups and a row is one contiguous bulk-copy target.
__device__ __forceinline__ constexpr uint32_t a_row_bytes(int K) { return (uint32_t)(K * 2 + 16); }
// Byte offset of 16-byte chunk `chunk` of row `row`.
__device__ __forceinline__ uint32_t a_chunk_off(int row, int chunk, int K) {
  return (uint32_t)row * a_row_bytes(K) + ((uint32_t)chunk << 4);
}

// A[16][K] <- src[T][K] (bf16, global); rows >= T are zero.  Lanes
// 0..T-1 of warp 0 each issue the bulk copy of one row (the bulk-copy
// engine moves the rows without tying up the load/store path); row r
// completes on BAR_SEG + r / kRowsPerSeg, so that work on the first rows can
// start while the later ones stream in.  seg_wait waits for the next row
// group, seg_finish for the rest and closes the staging.  Every compute
// thread calls these in the same order, after a barrier that ended the
// previous use of the staging area.
constexpr int kRowsPerSeg = kMaxT / kSegs;
static_assert(kRowsPerSeg * kSegs == kMaxT && kSegs < 8, "row groups of the staging");
__device__ __forceinline__ void stage_issue_inl(Ctx& c, const uint16_t* src, int K) {
  const int T = c.a()->dm.T;
  const int cpr = K / 8;
  uint8_t* Ag = c.smem() + kOffA;
  for (int row = T; row < kMaxT; ++row)
    for (int ch = c.tid(); ch < cpr; ch += kConsThreads)
      *reinterpret_cast<uint4*>(Ag + a_chunk_off(row, ch, K)) = make_uint4(0, 0, 0, 0);
  if (c.warp() == 0) {
    const uint32_t A = c.sbase() + kOffA;
    if (c.lane() < kSegs) {
      const int rows = min(max(T - c.lane() * kRowsPerSeg, 0), kRowsPerSeg);
      mbar_arrive_expect_tx(c.bar(BAR_SEG + c.lane()), (uint32_t)(rows * K * 2));
    }
    __syncwarp();
    if (c.lane() < T) {
      fence_proxy_async_shared();  // earlier generic accesses to the area before the copies' writes
      bulk_g2s(A + c.lane() * a_row_bytes(K), src + (size_t)c.lane() * K, (uint32_t)(K * 2),
               c.bar(BAR_SEG + c.lane() / kRowsPerSeg));
    }
  }
}

static __device__ __noinline__ void stage_issue(Ctx& c, const uint16_t* src, int K) { stage_issue_inl(c, src, K); }

// Waits (bounded, also after an abort: the copies must land before the
// block may exit) for the next row group of the current staging (c.sg % 8;
// the staging's barrier phase is c.sg / 8).
__device__ __forceinline__ void seg_wait(Ctx& c) {
  const bool ok = mbar_wait(c.bar(BAR_SEG + (c.sg & 7u)), (c.sg >> 3) & 1u, c.deadline(), &c.misc()->zero);
  if (!ok && !aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -4);
  c.sg++;
}

// Waits for every row group of the current staging up to `g`.
__device__ __forceinline__ void seg_wait_upto(Ctx& c, int g) {
  while ((int)(c.sg & 7u) <= g) seg_wait(c);
}

__device__ __forceinline__ void seg_finish(Ctx& c) {
  seg_wait_upto(c, kSegs - 1);
  c.sg = (c.sg | 7u) + 1u;
}

// Waits (bounded) for the latest query staging of the attention phase.
__device__ __forceinline__ bool stage_wait(Ctx& c) {
  const bool ok = mbar_wait(c.bar(BAR_STG), c.nstg & 1, c.deadline(), &c.misc()->zero);
  c.nstg++;
  if (!ok && !aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -4);
  return ok;
}

// A[16][K] <- rb(RMSNorm(src; gamma, eps)) per row.  With `partials`, the
// row statistics come from the per-block sums of squares that the residual
// projection which wrote `src` left in ss_part (summed here over the blocks
// in a fixed order, while the rows stream in), and each row group is scaled
// as soon as it lands; otherwise every block computes them from the staged
// rows in the same fixed order, once every row has landed.  Returns with
// every row group waited for (the staging stays open until the
// projection's seg_finish).
static_assert(kMaxK / 8 <= 2 * kConsThreads, "a thread scales at most two 8-element chunks of gamma");
static_assert(kMaxT <= 2 * kConsWarps, "a warp sums the partials of at most two tokens");
static __device__ __noinline__ void stage_rmsnorm(Ctx& c, const uint16_t* src, const uint16_t* gamma, int K,
                                                 bool partials) {
  const Dims& d = c.a()->dm;
  const int cpr = K / 8;
  // the (at most two) gamma chunks this thread scales, loaded while the rows stream in
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  const int ch0 = c.tid(), ch1 = c.tid() + kConsThreads;
  uint4 gv0 = make_uint4(0, 0, 0, 0), gv1 = make_uint4(0, 0, 0, 0);
  if (ch0 < cpr) gv0 = __ldg(g4 + ch0);
  if (ch1 < cpr) gv1 = __ldg(g4 + ch1);
  uint8_t* A = c.smem() + kOffA;
  if (partials) {
    // warp w: tokens 2w and 2w + 1; lane l sums blocks l, l + 32, ... in
    // order (up to 256 blocks per pass, every load of a pass in flight at
    // once; the partials are token-major, so each load instruction of a warp
    // reads consecutive words), then the lanes are folded by a fixed butterfly.
    // The first pass's loads are issued before the rows' bulk copies, so
    // that they do not queue behind the copies in L2: the statistics are
    // then known while the rows stream in.
    const float* ssp = c.a()->s.ss_part;
    float ss[2] = {0.f, 0.f};
    for (int p0 = 0; p0 < c.nctas(); p0 += 256) {
      float v[2][8];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int t = 2 * c.warp() + i, p = p0 + c.lane() + 32 * j;
          v[i][j] = (t < d.T && p < c.nctas()) ? __ldcg(ssp + (size_t)t * c.nctas() + p) : 0.f;
        }
      if (p0 == 0) stage_issue_inl(c, src, K);
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) ss[i] += v[i][j];
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
      const int t = 2 * c.warp() + i;
      if (t < d.T && c.lane() == 0) c.misc()->inv_rms[t] = 1.0f / sqrtf(ss[i] / (float)K + d.eps);
    }
    named_bar(1, kConsThreads);  // every row's statistic is known
  } else {
    stage_issue_inl(c, src, K);
    seg_wait_upto(c, kSegs - 1);
    named_bar(1, kConsThreads);
    // sum of squares: warp w owns rows w and w + 8
    for (int rr = 0; rr < 2; ++rr) {
      const int row = c.warp() + 8 * rr;
      float ss = 0.f;
      if (row < d.T) {
#pragma unroll 1
        for (int ch = c.lane(); ch < cpr; ch += 32) {
          const uint4 v = *reinterpret_cast<const uint4*>(A + a_chunk_off(row, ch, K));
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = bf16_lo(w[j]), hi = bf16_hi(w[j]);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (c.lane() == 0) c.misc()->inv_rms[row] = 1.0f / sqrtf(ss / (float)K + d.eps);
      }
    }
    named_bar(1, kConsThreads);
  }
  stamp(c, 47);
  const float* inv_rms = c.misc()->inv_rms;
  // row group by row group as they land: the thread's (at most two) chunks
  // of the group's rows, the group's loads of one chunk issued together; the
  // products (x inv) gamma are formed two at a time (f32x2, rounded like
  // two single multiplies)
  const int T = d.T, nch = ch1 < cpr ? 2 : (ch0 < cpr ? 1 : 0);
  const uint32_t rbytes = a_row_bytes(K);
  uint8_t* ap[2] = {A + ch0 * 16, A + ch1 * 16};
  uint64_t gp[2][4];
  {
    const uint32_t g0[4] = {gv0.x, gv0.y, gv0.z, gv0.w}, g1[4] = {gv1.x, gv1.y, gv1.z, gv1.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      gp[0][j] = f32x2_pack(bf16_lo(g0[j]), bf16_hi(g0[j]));
      gp[1][j] = f32x2_pack(bf16_lo(g1[j]), bf16_hi(g1[j]));
    }
  }
#pragma unroll 1
  for (int r0 = 0; r0 < T; r0 += kRowsPerSeg) {
    seg_wait_upto(c, r0 / kRowsPerSeg);
#pragma unroll 1
    for (int k = 0; k < nch; ++k) {
      uint64_t g[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) g[j] = k ? gp[1][j] : gp[0][j];
      uint8_t* const p = k ? ap[1] : ap[0];
      uint4 v[kRowsPerSeg];
#pragma unroll
      for (int i = 0; i < kRowsPerSeg; ++i) v[i] = *reinterpret_cast<const uint4*>(p + (r0 + i) * rbytes);
#pragma unroll
      for (int i = 0; i < kRowsPerSeg; ++i) {
        if (r0 + i >= T) break;
        const uint64_t inv = f32x2_pack(inv_rms[r0 + i], inv_rms[r0 + i]);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          o[j] = f32x2_to_bf16x2(f32x2_mul(f32x2_mul(f32x2_pack(bf16_lo(w[j]), bf16_hi(w[j])), inv), g[j]));
        *reinterpret_cast<uint4*>(p + (r0 + i) * rbytes) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  stamp(c, 51);
}

// Waits for ring tile `c.seq`; false on abort/timeout (the caller still
// releases the slot and advances).
__device__ __forceinline__ bool wait_tile(Ctx& c) {
  const uint32_t s = c.seq % kSlots;
  if (mbar_wait(c.bar(BAR_FULL + s), (c.seq / kSlots) & 1, c.deadline(), c.abort_ptr())) return true;
  if (!aborted(c)) raise_error(c, ERR_TIMEOUT_RING, -2);
  return false;
}

__device__ __forceinline__ void release_tile(Ctx& c) {
  __syncwarp();
  if (c.lane() == 0) mbar_arrive(c.bar(BAR_EMPTY + c.seq % kSlots));
  c.seq++;
}

// ---------------------------------------------------------------------------
// epilogues
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t ldcg32(const uint16_t* p) {
  return __ldcg(reinterpret_cast<const unsigned int*>(p));
}
__device__ __forceinline__ void st32(uint16_t* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }

// Global operands of a group's epilogue (residual values, router bias or
// RoPE cos / sin of the lane's two tokens), loaded before the group's
// products so that the epilogue adds no L2 round trip to the phase.
struct EpiPre {
  uint32_t r[4];
};

// out = rb(resid + rb(x W^T))  (h1 after the output projection, h2 after the
// unpooler); pre.r[h] = resid[g + 8 h][n .. n + 1].  Returns the sums of
// squares of the lane's two stored values of tokens g and g + 8 (the next
// RMSNorm's statistics).
struct EpiResidual {
  uint16_t* out;  // [T][D]
  int T, D;
  __device__ float2 operator()(int n0, int lane, const float* v, const EpiPre& pre) const {
    const int g = lane >> 2, n = n0 + 2 * (lane & 3);
    float ss[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = g + 8 * h;
      if (t >= T) continue;
      const uint32_t r = pre.r[h];
      const float a = bf16_round(v[2 * h]), b = bf16_round(v[2 * h + 1]);
      const uint32_t o = pack_bf16x2(bf16_lo(r) + a, bf16_hi(r) + b);
      st32(out + (size_t)t * D + n, o);
      ss[h] = bf16_lo(o) * bf16_lo(o) + bf16_hi(o) * bf16_hi(o);
    }
    return make_float2(ss[0], ss[1]);
  }
};

// out = rb(x W^T)
struct EpiStore {
  uint16_t* out;
  int T, N;
  __device__ void operator()(int n0, int lane, const float* v) const {
    const int g = lane >> 2, n = n0 + 2 * (lane & 3);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = g + 8 * h;
      if (t < T) st32(out + (size_t)t * N + n, pack_bf16x2(v[2 * h], v[2 * h + 1]));
    }
  }
};

// logits = fp32(pooled W_r^T) + bias; pre.r[0..1] = bias[n], bias[n + 1]
struct EpiRouter {
  float* out;
  int T, E;
  __device__ void operator()(int n0, int lane, const float* v, const EpiPre& pre) const {
    const int g = lane >> 2, n = n0 + 2 * (lane & 3);
    const float b0 = __uint_as_float(pre.r[0]), b1 = __uint_as_float(pre.r[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = g + 8 * h;
      if (t < T)
        *reinterpret_cast<float2*>(out + (size_t)t * E + n) = make_float2(v[2 * h] + b0, v[2 * h + 1] + b1);
    }
  }
};

// qkv = rb(x W_qkv^T); RoPE (rotate-half) on q and k; K, V rows into the
// cache at the verify positions; q into the stash.  Rows of q / k heads are
// stored pair-adjacent (i, i + d/2) in the tiled weight, so v[0], v[1] of a
// lane are one rotation pair.  pre.r[2h], pre.r[2h + 1] = cos, sin of the
// pair's angle for token g + 8 h (q and k rows).
struct EpiQKV {
  uint16_t* q_stash;  // [T][Hq][hd]
  uint16_t* kv;       // [2][Hkv][max_seq][hd] of the layer being written
  int T, Hq, Hkv, hd, max_seq, pos0;
  __device__ void operator()(int n0, int lane, const float* v, const EpiPre& pre) const {
    const int g = lane >> 2, n = n0 + 2 * (lane & 3);
    const int qk_rows = (Hq + Hkv) * hd;
    const int hs = 31 - __clz(hd);  // head_dim is a power of two
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = g + 8 * h;
      if (t >= T) continue;
      const float a = bf16_round(v[2 * h]), b = bf16_round(v[2 * h + 1]);
      if (n < qk_rows) {
        const int head = n >> hs, i = (n & (hd - 1)) >> 1;
        const float cs = __uint_as_float(pre.r[2 * h]), sn = __uint_as_float(pre.r[2 * h + 1]);
        const float ra = a * cs - b * sn;
        const float rbv = a * sn + b * cs;
        uint16_t* dst;
        if (head < Hq) {
          dst = q_stash + ((size_t)t * Hq + head) * hd;
        } else {
          dst = kv + ((size_t)(head - Hq) * max_seq + pos0 + t) * hd;
        }
        dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(ra));
        dst[i + hd / 2] = __bfloat16_as_ushort(__float2bfloat16_rn(rbv));
      } else {
        const int vr = n - qk_rows, kvh = vr >> hs, j = vr & (hd - 1);
        uint16_t* dst = kv + ((size_t)(Hkv + kvh) * max_seq + pos0 + t) * hd + j;
        st32(dst, pack_bf16x2(a, b));
      }
    }
  }
};

// The dense projections of a launch, each with its epilogue; the epilogue's
// operands are taken from the launch arguments (in shared memory) when it
// runs, so nothing about them lives in local memory.
enum DenseOp : int {
  OP_QKV_CUR = 0,  // this layer's QKV (launches that run the prologue)
  OP_OPROJ = 1,    // h1 = hidden + rb(o W_o^T)
  OP_POOL = 2,     // pooled = rb(RMSNorm(h1) W_pool^T)
  OP_ROUTER = 3,   // logits = pooled W_r^T + bias
  OP_UNPOOL = 4,   // hidden = h1 + rb(m W_unpool^T)
  OP_QKV_NXT = 5,  // the next layer's QKV and KV write
};

__device__ __forceinline__ bool op_residual(int op) { return op == OP_OPROJ || op == OP_UNPOOL; }

// Loads the global operands of op's epilogue for the row group at n0.
__device__ __forceinline__ EpiPre dense_epi_pre(const LaunchArgs& a, int op, int n0, int lane) {
  const Dims& d = a.dm;
  const int g = lane >> 2, n = n0 + 2 * (lane & 3);
  EpiPre p = {{0u, 0u, 0u, 0u}};
  if (op_residual(op)) {
    const uint16_t* resid = op == OP_OPROJ ? a.hidden : a.s.h1;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (g + 8 * h < d.T) p.r[h] = ldcg32(resid + (size_t)(g + 8 * h) * d.D + n);
  } else if (op == OP_ROUTER) {
    p.r[0] = __float_as_uint(__ldg(a.cur.router_bias + n));
    p.r[1] = __float_as_uint(__ldg(a.cur.router_bias + n + 1));
  } else if (op == OP_QKV_CUR || op == OP_QKV_NXT) {
    if (n < (d.Hq + d.Hkv) * d.hd) {
      const int i = (n & (d.hd - 1)) >> 1;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if (g + 8 * h < d.T) {
          const float2 cs = __ldcg(reinterpret_cast<const float2*>(a.s.rope + ((size_t)(g + 8 * h) * (d.hd / 2) + i) * 2));
          p.r[2 * h] = __float_as_uint(cs.x);
          p.r[2 * h + 1] = __float_as_uint(cs.y);
        }
    }
  }
  return p;
}

// Runs op's epilogue; for the residual ops, returns the lane's sums of
// squares of tokens g and g + 8 (zeros otherwise).
__device__ __forceinline__ float2 dense_epilogue(const LaunchArgs& a, int op, int n0, int lane, const float* v,
                                                 const EpiPre& pre) {
  const Dims& d = a.dm;
  if (op_residual(op)) return EpiResidual{op == OP_OPROJ ? a.s.h1 : a.hidden, d.T, d.D}(n0, lane, v, pre);
  if (op == OP_POOL) EpiStore{a.s.pooled, d.T, d.P}(n0, lane, v);
  else if (op == OP_ROUTER) EpiRouter{a.s.logits, d.T, d.E}(n0, lane, v, pre);
  else EpiQKV{a.s.q_stash, op == OP_QKV_CUR ? a.kv_cur : a.kv_nxt, d.T, d.Hq, d.Hkv, d.hd, d.max_seq, a.pos0}(n0, lane, v, pre);
  return make_float2(0.f, 0.f);
}

// Dense projection out[t][n] = sum_k A[t][k] W[n][k] over this block's row
// groups.  Each 16 KB tile is split along K across the 8 warps; per-group
// partial sums are reduced in a fixed warp order and handed to `epi` by a
// rotating warp (so the others keep consuming tiles).
//   epilogue(n0, lane, v[4]): v = {D[g][n0+2c], D[g][n0+2c+1], D[g+8][n0+2c],
//   D[g+8][n0+2c+1]} with g = lane / 4, c = lane % 4.
// The epilogues run one group at a time in group order (each is ordered
// before the next group's reduction barrier), so the residual ops fold their
// rows' sums of squares into the block's ssq[] without races and in a fixed
// order; the block's totals go to ss_part[t][cta] at the end of the phase.
static __device__ __noinline__ void dense_phase(Ctx& cin, const uint8_t* wbase, int N, int K, int op) {
  const int tslot = kSlotDense + 4 * op;
  Ctx c = cin;  // register copy of the ring position (written back at exit)
  const DenseSched s = dense_sched(wbase, N, K, c.cta(), c.nctas());
  const int nkb = s.tb / 512;  // 32-wide K blocks per tile
  const int kb0 = c.warp() * nkb / kConsWarps, kb1 = (c.warp() + 1) * nkb / kConsWarps;
  const uint32_t A = c.sbase() + kOffA;
  const int arow = c.lane() & 15;
  const uint32_t a_row_base = A + arow * a_row_bytes(K);
  float* red = reinterpret_cast<float*>(c.smem() + kOffRed);
  const bool resid = op_residual(op);
  if (resid && c.tid() < kMaxT) c.misc()->ssq[c.tid()] = 0.f;
  // warp w runs the epilogues of groups w, w + 8, ...: the first one's
  // operands are loaded now, in flight while the products are formed
  EpiPre pre = {{0u, 0u, 0u, 0u}};
  if (c.warp() < s.ng) pre = dense_epi_pre(*c.a(), op, 8 * (s.g0 + c.warp()), c.lane());
  stamp(c, tslot);
  for (int gi = 0; gi < s.ng; ++gi) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int part = 0; part < s.tpg; ++part) {
      const bool ok = wait_tile(c);
      if (gi == 0 && part == 0) seg_wait_upto(c, kSegs - 1);  // every row of the staging
      if (gi == 0 && part == 0) stamp(c, tslot + 1);
      if (ok) {
        const uint32_t slot = c.slot_addr(c.seq % kSlots);
        const int kbase = part * (s.tb / 16);
        if (kb1 - kb0 == 4) {
          // a full tile's share (four K blocks): every shared-memory load
          // issued before the first product, so their latencies overlap
          const uint32_t bp = slot + kb0 * 512 + c.lane() * 16;
          const uint32_t ap = a_row_base + ((((kbase + kb0 * 32) >> 3) + (c.lane() >> 4)) << 4);
          uint4 b[4];
          uint32_t a[8][4];
#pragma unroll
          for (int q = 0; q < 4; ++q) b[q] = lds128(bp + q * 512);
#pragma unroll
          for (int q = 0; q < 8; ++q) ldmatrix_x4(a[q], ap + q * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            mma_bf16(acc, a[2 * q], b[q].x, b[q].y);
            mma_bf16(acc, a[2 * q + 1], b[q].z, b[q].w);
          }
        } else {
          for (int kb = kb0; kb < kb1; ++kb) {
            const uint4 b = lds128(slot + kb * 512 + c.lane() * 16);
            const int k0 = kbase + kb * 32;
            uint32_t a[4];
            ldmatrix_x4(a, a_row_base + (((k0 >> 3) + (c.lane() >> 4)) << 4));
            mma_bf16(acc, a, b.x, b.y);
            ldmatrix_x4(a, a_row_base + (((k0 >> 3) + 2 + (c.lane() >> 4)) << 4));
            mma_bf16(acc, a, b.z, b.w);
          }
        }
      }
      release_tile(c);
    }
    float* rb_ = red + (gi & 1) * (kConsWarps * 32 * 4);
    *reinterpret_cast<float4*>(rb_ + (c.warp() * 32 + c.lane()) * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    named_bar(1, kConsThreads);
    if (c.warp() == (gi & (kConsWarps - 1))) {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < kConsWarps; ++w) {
        const float4 p = *reinterpret_cast<const float4*>(rb_ + (w * 32 + c.lane()) * 4);
        v[0] += p.x;
        v[1] += p.y;
        v[2] += p.z;
        v[3] += p.w;
      }
      // (one decision per warp: the shuffles below need every lane)
      if (__shfl_sync(0xffffffffu, (int)aborted(c), 0) == 0) {
        if (gi >= kConsWarps) pre = dense_epi_pre(*c.a(), op, 8 * (s.g0 + gi), c.lane());
        float2 ss = dense_epilogue(*c.a(), op, 8 * (s.g0 + gi), c.lane(), v, pre);
        if (resid) {
          ss.x += __shfl_xor_sync(0xffffffffu, ss.x, 1);
          ss.x += __shfl_xor_sync(0xffffffffu, ss.x, 2);
          ss.y += __shfl_xor_sync(0xffffffffu, ss.y, 1);
          ss.y += __shfl_xor_sync(0xffffffffu, ss.y, 2);
          if ((c.lane() & 3) == 0) {
            c.misc()->ssq[c.lane() >> 2] += ss.x;
            c.misc()->ssq[(c.lane() >> 2) + 8] += ss.y;
          }
        }
      }
    }
  }
  if (resid) {
    named_bar(1, kConsThreads);
    if (c.tid() < kMaxT) c.a()->s.ss_part[(size_t)c.tid() * c.nctas() + c.cta()] = c.misc()->ssq[c.tid()];
  }
  seg_finish(c);  // (a block without row groups waits for the staging here)
  stamp(c, tslot + 2);
  cin = c;
}

// cos / sin of p * theta^(-2i/d) for the step's positions (p = cached
// length + the slot's depth in the candidate tree; S + t for the chain).  The inverse
// frequencies theta^(-2i/d) are a model constant (computed once in double
// at model creation); the angle p * inv_freq is formed and reduced to
// [-pi, pi] in double, then rounded once to float for the sine / cosine.
static __device__ __noinline__ void rope_table(Ctx& c) {
  const Dims& d = c.a()->dm;
  const int half = d.hd / 2, n = d.T * half;
  for (int e = c.cta() * kConsThreads + c.tid(); e < n; e += c.nctas() * kConsThreads) {
    const int t = e / half, i = e % half;
    const double ang = (double)(c.a()->pos0 + c.a()->depth[t]) * c.a()->s.inv_freq[i];
    const double two_pi = 6.283185307179586476925286766559;
    const double r = ang - rint(ang * (1.0 / two_pi)) * two_pi;
    float sn, cs;
    __sincosf((float)r, &sn, &cs);
    c.a()->s.rope[2 * e] = cs;
    c.a()->s.rope[2 * e + 1] = sn;
  }
}

// ---------------------------------------------------------------------------
// attention: split-KV over (kv head, key range) units, one per block
// ---------------------------------------------------------------------------

// Key splits per kv head: one block each, at most 32 (the combine keeps
// split s in lane s), at least 16 keys per split.
__device__ __forceinline__ int attn_splits(const Dims& d, int nkeys, int nctas) {
  int ns = min(min(nctas / d.Hkv, 32), (nkeys + 15) / 16);
  return ns < 1 ? 1 : ns;
}

__device__ __forceinline__ int attn_lo(const LaunchArgs& a) {
  return a.cur.window > 0 ? max(0, a.pos0 - a.cur.window + 1) : 0;
}

// KV stage layout: the K rows then the V rows of kAttnChunk keys, each as
// HD / 64 boxes of [kAttnChunk rows][128 bytes] (64 columns) written by the
// tiled copies with 128-byte swizzle: 16-byte piece u of a box row r sits at
// u ^ (r % 8), so the 8 rows an ldmatrix reads at one column fall in 8
// different bank groups.
constexpr uint32_t kKvBoxBytes = kAttnChunk * 128;
template <int HD>
__device__ __forceinline__ constexpr uint32_t kv_stage_bytes() { return 2u * (HD / 64) * kKvBoxBytes; }
// Byte offset of 16-byte piece q (columns 8 q .. 8 q + 7) of row r in a K or
// V area, for a lane whose row has r % 8 == sw.
__device__ __forceinline__ uint32_t kv_piece(int r, int q, int sw) {
  return (uint32_t)((q >> 3) * kKvBoxBytes + r * 128 + (((q & 7) ^ sw) << 4));
}

// Compute thread 0: the tiled copies of chunk ci's K and V rows (keys
// ks + ci kAttnChunk ..., a whole box each: rows past the split belong to
// the next split, rows past the cache are zero-filled) into stage
// ci % kAttnStages, completing on its barrier.  Called once every thread
// is done with the stage's previous contents.
template <int HD>
static __device__ __forceinline__ void attn_issue(Ctx& c, int ci, int nchunks, int h, int ks) {
  if (ci >= nchunks) return;
  const LaunchArgs& a = *c.a();
  const int st = ci % kAttnStages;
  const uint32_t kst = c.sbase() + kOffA + st * kv_stage_bytes<HD>();
  const uint32_t vst = kst + (HD / 64) * kKvBoxBytes;
  const uint32_t bar = c.bar(BAR_KV + st);
  const int j0 = ks + ci * kAttnChunk;
  fence_proxy_async_shared();  // earlier generic accesses to the stage before the copies' writes
  mbar_arrive_expect_tx(bar, kv_stage_bytes<HD>());
  const unsigned long long map = c.misc()->kvmap;
  // the cached rows are read once per step: evict_first, so that a long
  // cache does not push the kernel's code and the prefetched lines out of L2
  const uint64_t pol = policy_evict_first();
#pragma unroll
  for (int bx = 0; bx < HD / 64; ++bx) {
    tma_load_3d_hint(kst + bx * kKvBoxBytes, map, 64 * bx, j0, a.kv_z0 + h, bar, pol);
    tma_load_3d_hint(vst + bx * kKvBoxBytes, map, 64 * bx, j0, a.kv_z0 + a.dm.Hkv + h, bar, pol);
  }
}

template <int HD>
static __device__ __noinline__ void attention_phase(Ctx& c) {
  static_assert(HD % 64 == 0 && kAttnStages * 2 * (HD / 64) * kKvBoxBytes <= kABytes, "KV stages exceed the staging area");
  static_assert(kAttnChunk % 16 == 0 && kAttnChunk <= 256, "a KV chunk is whole 16-key blocks and one box high");
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  const int T = d.T, G = d.Hq / d.Hkv, GT = G * T;
  const int lo_all = attn_lo(a);
  const int nkeys = a.pos0 + T - lo_all;
  const int ns = attn_splits(d, nkeys, c.nctas());
  if (c.cta() >= ns * d.Hkv) return;  // uniform per block
  // the swizzled tiled copies need 1 KB aligned stages (a block-uniform test)
  if ((c.sbase() & 1023u) != 0u) {
    if (c.tid() == 0) raise_error(c, ERR_TIMEOUT_RING, -6);
    return;
  }
  const int h = c.cta() / ns, sp = c.cta() % ns;
  const int ks = lo_all + (int)((long long)sp * nkeys / ns);
  const int ke = lo_all + (int)((long long)(sp + 1) * nkeys / ns);
  const int n_mt = GT <= 16 ? 1 : (GT <= 32 ? 2 : 4);
  const int nparts = kConsWarps / n_mt;
  const int mt = c.warp() % n_mt, part = c.warp() / n_mt;
  const int g = c.lane() >> 2, cq = c.lane() & 3;
  const int W = a.cur.window;

  // my two rows: r = mt*16 + g (+8); row r -> (gq = r / T, t = r % T).
  // Token t (position pos0 + depth) sees the cached keys j < pos0 inside its
  // window and the verify keys pos0 + u of the slots u set in vis[t] (its
  // ancestors and itself in the candidate tree, already limited to the
  // window; u <= t for the chain).
  // Keys outside [plo, phi] are never visible (phi = the last verify slot
  // the row sees); inside, only a key block that reaches the verify rows
  // also tests the slot bits (a warp-uniform branch).
  int rows[2], plo[2], phi[2];
  uint32_t vmask[2];
  bool rv[2];
  for (int i = 0; i < 2; ++i) {
    rows[i] = mt * 16 + g + 8 * i;
    rv[i] = rows[i] < GT;
    const int t = rv[i] ? rows[i] % T : 0;
    plo[i] = W > 0 ? a.pos0 + a.depth[t] - W + 1 : 0;
    vmask[i] = rv[i] ? a.vis[t] : 0u;
    phi[i] = a.pos0 + 31 - __clz(vmask[i] | 1u);
  }
  const int pos0 = a.pos0;
  const int nchunks = (ke - ks + kAttnChunk - 1) / kAttnChunk;
  // Every compute thread loads its share of the head group's queries (T
  // runs of G x HD bf16, one per token; at most 4 16-byte pieces a thread,
  // their loads in flight together) into the last KV stage; compute thread 0
  // issues chunk 0 right behind its own query loads, and chunks 1 ..
  // kAttnStages - 2 once the queries are in (requested all at once, the
  // chunks' copies would hold the query loads up in the memory system).
  // The A fragments are read from the last stage, which is then handed to
  // chunk kAttnStages - 1.
  static_assert(64 * 128 / 8 <= 4 * kConsThreads, "query pieces per thread (G T <= 64 rows, HD <= 128)");
  const uint32_t qs = c.sbase() + kOffA + (kAttnStages - 1) * kv_stage_bytes<HD>();
  {
    constexpr int ppt = HD / 8;  // 16-byte pieces per query row
    const int prun = G * ppt, npieces = T * prun;
    uint4 qv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = c.tid() + u * kConsThreads;
      if (i < npieces)
        qv[u] = __ldcg(reinterpret_cast<const uint4*>(a.s.q_stash + ((size_t)(i / prun) * d.Hq + h * G) * HD) +
                       i % prun);
    }
    if (c.tid() == 0) attn_issue<HD>(c, 0, nchunks, h, ks);
    uint8_t* qg = c.smem() + kOffA + (kAttnStages - 1) * kv_stage_bytes<HD>();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = c.tid() + u * kConsThreads;
      if (i < npieces) *reinterpret_cast<uint4*>(qg + (size_t)i * 16) = qv[u];
    }
  }
  named_bar(1, kConsThreads);
  stamp(c, 55);
  if (c.tid() == 0)
    for (int ci = 1; ci < kAttnStages - 1; ++ci) attn_issue<HD>(c, ci, nchunks, h, ks);
  uint32_t qa[HD / 16][4];
  {
    // ldmatrix: lane l gives row l % 16 of the warp's 16-row tile, column
    // half l / 16; rows past G T read row 0 and are zeroed below
    const int r = mt * 16 + (c.lane() & 15), rr = r < GT ? r : 0;
    const uint32_t qrow = qs + (uint32_t)(((rr % T) * G + rr / T) * (HD * 2)) + ((c.lane() >> 4) << 4);
#pragma unroll
    for (int k = 0; k < HD / 16; ++k) {
      ldmatrix_x4(qa[k], qrow + k * 32);
      if (!rv[0]) qa[k][0] = qa[k][2] = 0u;
      if (!rv[1]) qa[k][1] = qa[k][3] = 0u;
    }
  }
  named_bar(1, kConsThreads);  // every warp has its fragments: the last stage is free
  if (c.tid() == 0) attn_issue<HD>(c, kAttnStages - 1, nchunks, h, ks);
  float o[HD / 8][4];
#pragma unroll
  for (int j = 0; j < HD / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float mrow[2] = {-CUDART_INF_F, -CUDART_INF_F}, lrow[2] = {0.f, 0.f};
  const float sl2 = rsqrtf((float)HD) * 1.4426950408889634f;
  const int sw = c.lane() & 7;  // the swizzle of every row this lane addresses

  for (int ci = 0; ci < nchunks; ++ci) {
    const int st = ci % kAttnStages;
    const int j0 = ks + ci * kAttnChunk;
    const int nrows = min(kAttnChunk, ke - j0);
    const int nblk = (nrows + 15) / 16;
    const uint32_t kst = c.sbase() + kOffA + st * kv_stage_bytes<HD>();
    const uint32_t vst = kst + (HD / 64) * kKvBoxBytes;
    // (bounded; also after an abort: the copies must land before the stage
    // is reused or the block exits)
    if (!mbar_wait(c.bar(BAR_KV + st), (uint32_t)(ci / kAttnStages) & 1u, c.deadline(), &c.misc()->zero) &&
        !aborted(c))
      raise_error(c, ERR_TIMEOUT_RING, -5);
    if (ci == 0) stamp(c, 62);
    if (ci == 1) stamp(c, 35);
    if (nrows < 16 * nblk) {
      // V rows past the split's last key up to its 16-key block: their P is
      // zero, but cache rows past the valid keys may hold non-finite values
      uint8_t* vz = c.smem() + kOffA + st * kv_stage_bytes<HD>() + (HD / 64) * kKvBoxBytes;
      const int nz = (16 * nblk - nrows) * 8;  // 16-byte pieces per box
      for (int i = c.tid(); i < nz * (HD / 64); i += kConsThreads) {
        const int bx = i / nz, rem = i % nz;
        *reinterpret_cast<uint4*>(vz + bx * kKvBoxBytes + (nrows + rem / 8) * 128 + (rem % 8) * 16) =
            make_uint4(0, 0, 0, 0);
      }
      named_bar(1, kConsThreads);
    }
    const bool ok = !aborted(c);
    for (int b = part; ok && b < nblk; b += nparts) {
      const int kb = j0 + 16 * b;
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      // S = Q K^T: ldmatrix rows = keys
      const int kr = 16 * b + (c.lane() & 7) + ((c.lane() >> 4) << 3), kpc = (c.lane() >> 3) & 1;
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        uint32_t kf[4];
        ldmatrix_x4(kf, kst + kv_piece(kr, 2 * k + kpc, sw));
        mma_bf16(sc[0], qa[k], kf[0], kf[1]);
        mma_bf16(sc[1], qa[k], kf[2], kf[3]);
      }
      float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
      const bool tail = kb + 16 > pos0;  // the block holds verify keys
      // a block of cached keys inside every row's window is visible to all
      // of the warp's rows: no per-key tests (a warp-uniform branch)
      const bool all_vis =
          __all_sync(0xffffffffu, !tail && kb + 16 <= ke && rv[0] && rv[1] && kb >= plo[0] && kb >= plo[1]);
      if (all_vis) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sc[nt][e] *= sl2;
            mx[e >> 1] = fmaxf(mx[e >> 1], sc[nt][e]);
          }
      } else {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int ri = e >> 1;
            const int key = kb + 8 * nt + 2 * cq + (e & 1);
            bool vis = rv[ri] && key < ke && key >= plo[ri] && key <= phi[ri];
            if (tail) vis = vis && (key < pos0 || ((vmask[ri] >> (key - pos0)) & 1u) != 0u);
            const float s = vis ? sc[nt][e] * sl2 : -CUDART_INF_F;
            sc[nt][e] = s;
            mx[ri] = fmaxf(mx[ri], s);
          }
      }
      float alpha[2], mu[2];
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 1));
        mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 2));
        const float mn = fmaxf(mrow[ri], mx[ri]);
        mu[ri] = mn == -CUDART_INF_F ? 0.f : mn;
        alpha[ri] = exp2f(mrow[ri] - mu[ri]);
        mrow[ri] = mn;
      }
      float ps[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ri = e >> 1;
          const float p = exp2f(sc[nt][e] - mu[ri]);
          sc[nt][e] = p;
          ps[ri] += p;
        }
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        ps[ri] += __shfl_xor_sync(0xffffffffu, ps[ri], 1);
        ps[ri] += __shfl_xor_sync(0xffffffffu, ps[ri], 2);
        lrow[ri] = lrow[ri] * alpha[ri] + ps[ri];
      }
      // rescale only when some row's running maximum moved (alpha == 1
      // otherwise, and the products would be the values themselves)
      if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int j = 0; j < HD / 8; ++j) {
          o[j][0] *= alpha[0];
          o[j][1] *= alpha[0];
          o[j][2] *= alpha[1];
          o[j][3] *= alpha[1];
        }
      }
      // P as bf16 hi + lo parts (P = hi + lo to ~16 significant bits), so
      // the P V product keeps fp32-level accuracy on the tensor cores.
      uint32_t pa[4], pl[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float x0 = sc[q >> 1][2 * (q & 1)], x1 = sc[q >> 1][2 * (q & 1) + 1];
        pa[q] = pack_bf16x2(x0, x1);
        pl[q] = pack_bf16x2(x0 - bf16_lo(pa[q]), x1 - bf16_hi(pa[q]));
      }
      // O += P V: ldmatrix.trans rows = keys
      const int vr = 16 * b + (c.lane() & 7) + (((c.lane() >> 3) & 1) << 3), vpc = c.lane() >> 4;
#pragma unroll
      for (int n0 = 0; n0 < HD / 16; ++n0) {
        uint32_t vf[4];
        ldmatrix_x4_trans(vf, vst + kv_piece(vr, 2 * n0 + vpc, sw));
        mma_bf16(o[2 * n0], pa, vf[0], vf[1]);
        mma_bf16(o[2 * n0 + 1], pa, vf[2], vf[3]);
        mma_bf16(o[2 * n0], pl, vf[0], vf[1]);
        mma_bf16(o[2 * n0 + 1], pl, vf[2], vf[3]);
      }
    }
    named_bar(1, kConsThreads);  // everyone is done with stage st
    if (c.tid() == 0) attn_issue<HD>(c, ci + kAttnStages, nchunks, h, ks);
  }
  stamp(c, 63);

  // merge the nparts key partitions of each 16-row tile through shared
  // memory (rows padded to HD + 4 floats), four threads per row, then write
  // this block's partial (unnormalised O, running max and sum in the log2
  // domain); per row the partitions are folded in ascending order
  constexpr int HDP = HD + 4;
  float* mb = reinterpret_cast<float*>(c.smem() + kOffA);  // [8][16][HDP]
  float* mlb = mb + kConsWarps * 16 * HDP;                // [8][16][2]
  {
    float* my = mb + c.warp() * 16 * HDP;
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) {
      const int col = 8 * j + 2 * cq;
      *reinterpret_cast<float2*>(my + g * HDP + col) = make_float2(o[j][0], o[j][1]);
      *reinterpret_cast<float2*>(my + (g + 8) * HDP + col) = make_float2(o[j][2], o[j][3]);
    }
    if (cq == 0) {
      mlb[(c.warp() * 16 + g) * 2] = mrow[0];
      mlb[(c.warp() * 16 + g) * 2 + 1] = lrow[0];
      mlb[(c.warp() * 16 + g + 8) * 2] = mrow[1];
      mlb[(c.warp() * 16 + g + 8) * 2 + 1] = lrow[1];
    }
  }
  named_bar(1, kConsThreads);
  stamp(c, 39);
  // thread (r, q) of the kTpr threads of row r takes the 4-column pieces
  // q, q + kTpr, ...: the kTpr threads of a row read and write contiguous
  // 16 kTpr-byte runs, so that each store instruction fills whole sectors
  constexpr int kTpr = kConsThreads / 64, kCpt = HD / kTpr;  // threads per row, columns per thread
  const int r = c.tid() / kTpr, cs = (c.tid() % kTpr) * 4;
  if (r < GT && !aborted(c)) {
    const int rmt = r >> 4, r16 = r & 15;
    float M = -CUDART_INF_F;
    for (int p = 0; p < nparts; ++p) M = fmaxf(M, mlb[((p * n_mt + rmt) * 16 + r16) * 2]);
    const float Mu = M == -CUDART_INF_F ? 0.f : M;
    float L = 0.f;
    float acc[kCpt];
#pragma unroll
    for (int j = 0; j < kCpt; ++j) acc[j] = 0.f;
    for (int p = 0; p < nparts; ++p) {
      const int w = (p * n_mt + rmt) * 16 + r16;
      const float wt = exp2f(mlb[w * 2] - Mu);
      L += wt * mlb[w * 2 + 1];
      const float* src = mb + w * HDP + cs;
#pragma unroll
      for (int j = 0; j < kCpt; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(src + j * kTpr);
        acc[j] += wt * v.x;
        acc[j + 1] += wt * v.y;
        acc[j + 2] += wt * v.z;
        acc[j + 3] += wt * v.w;
      }
    }
    float* op = a.s.o_part + ((size_t)c.cta() * 64 + r) * HD + cs;
#pragma unroll
    for (int j = 0; j < kCpt; j += 4)
      *reinterpret_cast<float4*>(op + j * kTpr) = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
    if (cs == 0) {
      float* mlp = a.s.ml_part + ((size_t)c.cta() * 64 + r) * 2;
      mlp[0] = M;
      mlp[1] = L;
    }
  }
  stamp(c, 43);
}

// o[t][(h G + gq) d + i] = rb(sum_s w_s O_s / sum_s w_s l_s), w_s = 2^(m_s - M)
// Work item = (kv head, row, 64-column slice): a warp, lane c = columns 2c
// and 2c + 1 of the slice, so that the 1,024 items of the full head shape
// give every warp of the grid at most one.  Lane s holds split s's (m, l);
// every split's values are loaded at once with the maxima (one L2 round
// trip) and summed over s in ascending order.
template <int HD>
static __device__ __noinline__ void combine_phase(Ctx& c) {
  const LaunchArgs& a = *c.a();
  const Dims& d = a.dm;
  const int T = d.T, G = d.Hq / d.Hkv, GT = G * T;
  const int nkeys = a.pos0 + T - attn_lo(a);
  const int ns = attn_splits(d, nkeys, c.nctas());  // <= 32: split s sits in lane s
  constexpr int kSlices = HD / 64;
  const int nitems = d.Hkv * GT * kSlices;
  const int sl = min(c.lane(), ns - 1);
#pragma unroll 1
  for (int it = c.cta() * kConsWarps + c.warp(); it < nitems; it += c.nctas() * kConsWarps) {
    const int pr = it / kSlices, col = (it % kSlices) * 64 + 2 * c.lane();
    const int h = pr / GT, r = pr % GT;
    const float* mlh = a.s.ml_part + ((size_t)h * ns * 64 + r) * 2;        // split s at + 128 s
    const float* oph = a.s.o_part + ((size_t)h * ns * 64 + r) * HD + col;  // split s at + 64 HD s
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(mlh + (size_t)sl * 128));
    float2 ov[32];
#pragma unroll
    for (int k = 0; k < 32; ++k)  // (clamped: in bounds; splits past ns weigh 0)
      ov[k] = __ldcg(reinterpret_cast<const float2*>(oph + min(k, ns - 1) * (64 * HD)));
    float M = c.lane() < ns ? ml.x : -CUDART_INF_F;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float Mu = M == -CUDART_INF_F ? 0.f : M;
    const float w = c.lane() < ns ? exp2f(ml.x - Mu) : 0.f;
    const float wl = w * ml.y;
    // (splits past ns add exact zeros: their weight is 0 and their values finite)
    float acc0 = 0.f, acc1 = 0.f, L = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float ws = __shfl_sync(0xffffffffu, w, k), ls = __shfl_sync(0xffffffffu, wl, k);
      L += ls;
      acc0 += ws * ov[k].x;
      acc1 += ws * ov[k].y;
    }
    const float inv = 1.0f / L;
    *reinterpret_cast<uint32_t*>(a.s.attn_o + (size_t)(r % T) * d.Hq * HD + (size_t)(h * G + r / T) * HD + col) =
        pack_bf16x2(acc0 * inv, acc1 * inv);
  }
}

}  // namespace msk
