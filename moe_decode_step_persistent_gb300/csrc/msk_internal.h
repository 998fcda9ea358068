// Internal definitions shared by the host launcher and the kernels.
//
// Library-owned HBM layouts (built by msk_load_layer):
//
//  Dense bf16 matrix W[N][K] ("tiled dense"): rows in groups of 8; each
//  group is K/32 fragment blocks of 512 bytes, and lane l = 4g + c of a
//  block holds W[8i + g][32b + {2c, 2c+1, 2c+8, 2c+9, 16+2c, 17+2c, 24+2c,
//  25+2c}] (8 bf16): exactly the B operands of two m16n8k16 mma steps.
//  Group i occupies bytes [16 K i, 16 K (i+1)).  CTA c of P reads the
//  contiguous groups [c*NG/P, (c+1)*NG/P).  The QKV matrix is stored with
//  rows (i, i + d/2) of every q and k head adjacent, so one lane holds both
//  members of a RoPE pair.
//
//  NVFP4 expert e ("tiled expert", expert_bytes(P, I) bytes each):
//    [GEMM1 units: I/16 of them][GEMM2 units: P/16 of them]
//  A GEMM1 unit covers 16 intermediate rows of gate and up (two row groups
//  of 8 each).  Its tiles, in order, for each K half kh (kchunks of 128
//  elements, at most 8 per tile): gate(kh) then up(kh); a tile holds, for
//  each of its two row groups, nk blocks of 576 bytes: 512 bytes of codes
//  (lane l = 4g + c holds 16 bytes: for k16 step s = 0..7 the bytes with
//  elements {16s+2c, 16s+2c+1} and {16s+2c+8, 16s+2c+9} of row g) and 64
//  bytes of block scales (row g's 8 E4M3 scales at offset 8g).
//  A GEMM2 unit covers 16 output rows of down (two row groups), same block
//  format, tiles of at most 8 kchunks.
#pragma once

#include <cstddef>
#include <cstdint>

#ifdef __CUDACC__
#define MSK_HD __host__ __device__
#else
#define MSK_HD
#endif

namespace msk {

constexpr int kConsWarps = 8;                    // compute warps per CTA
constexpr int kConsThreads = 32 * kConsWarps;    // 256
constexpr int kThreads = kConsThreads + 32;      // + one producer warp
constexpr int kSlotBytes = 16384;                // weight ring slot
constexpr int kSlots = 5;                        // ring depth (80 KB)
constexpr int kMaxT = 16;                        // verify tokens
constexpr int kMaxK = 4096;                      // widest dense input
constexpr int kABytes = kMaxT * (kMaxK * 2 + 16);  // activation staging area (rows padded by 16 bytes)
constexpr int kBlk4 = 576;                       // NVFP4 bytes per 8 rows x k128
constexpr int kTile4 = 2 * kBlk4;                // NVFP4 tile: 16 rows x k128 (1152 B)
constexpr int kAttnChunk = 112;                  // keys per KV stage
constexpr int kTimelineSlots = 64;
// Timeline slots: [0, PH_COUNT) phase starts; 14 top-k chosen; 15 dispatch
// ready; 16 + phase: the block's work in a phase done; kSlotDense + 4 k +
// {0: entry (activations staged), 1: first weight tile in, 2: last group's
// products done} for the k-th dense projection of the launch; 30, 31: warp
// 0's logits loaded / top-k rounds done; 62, 63: attention's first KV chunk
// landed / key loop done.
constexpr int kSlotDense = 32;
// kSlotExpert + {0: GEMM1 activations staged, 1: warp 0's first step done,
// 2: warp 0's units done, 3..5: the same for GEMM2}
constexpr int kSlotExpert = 56;

// phases of one launch (timeline slots, error reports)
enum Phase : int {
  PH_START = 0,
  PH_PRO_QKV,
  PH_ATTN,
  PH_COMBINE,
  PH_OPROJ,
  PH_POOL,
  PH_ROUTER,
  PH_TOPK,
  PH_GEMM1,
  PH_GEMM2,
  PH_MCOMB,  // (fused into GEMM2; slot kept for timeline numbering)
  PH_UNPOOL,
  PH_QKV,
  PH_END,
  PH_COUNT
};

MSK_HD inline constexpr size_t dense_tiled_bytes(int64_t N, int64_t K) { return (size_t)N * K * 2; }
// NVFP4 tile (16 weight rows r x k128, the mma A operand of eight k16
// steps): bytes [0, 1024) codes, lane-major in two halves: byte
// 512 h + 16 L + 4 (s - 4 h) + j for lane L = 4 g + c, k16 step s (half
// h = s / 4) and register j = 2 k8 + r8 holds the E2M1 pair of row
// g + 8 r8, columns 16 s + 8 k8 + 2 c (low nibble) and + 1 (high nibble);
// bytes [1024, 1152) the E4M3 scales, [16 rows][8 k16 blocks].
MSK_HD inline constexpr int tile4_code_off(int r, int k) {
  return 512 * ((k >> 4) >> 2) + 16 * (4 * (r & 7) + ((k & 7) >> 1)) + 4 * ((k >> 4) & 3) +
         (2 * ((k >> 3) & 1) + ((r >> 3) & 1));
}
MSK_HD inline constexpr int tile4_scale_off(int r, int k) { return 1024 + 8 * r + (k >> 4); }
// GEMM1 unit: 16 intermediate rows of gate and up, all of K, ordered
// [k128 chunk][gate, up] tiles.  GEMM2 unit: 32 output rows of down, all of
// K, ordered [k128 chunk][rows 0-15, rows 16-31].  A streaming step of
// consecutive chunks is one contiguous range.
constexpr int kG1Rows = 16;
constexpr int kG2Rows = 32;
MSK_HD inline constexpr int g1_unit_bytes(int P) { return 2 * (P / 128) * kTile4; }
MSK_HD inline constexpr int g2_unit_bytes(int I) { return 2 * (I / 128) * kTile4; }
MSK_HD inline constexpr int g1_tile_off(int kc, int gu) { return (2 * kc + gu) * kTile4; }
MSK_HD inline constexpr int g2_tile_off(int kc, int half) { return (2 * kc + half) * kTile4; }
MSK_HD inline constexpr size_t expert_g1_bytes(int P, int I) { return (size_t)(I / kG1Rows) * g1_unit_bytes(P); }
MSK_HD inline constexpr size_t expert_bytes(int P, int I) {
  return expert_g1_bytes(P, I) + (size_t)(P / kG2Rows) * g2_unit_bytes(I);
}

struct Dims {
  int D, Hq, Hkv, hd, P, E, topk, I, T, max_seq, n_layers, pf_experts, nctas;
  float eps, theta;
};

// One layer on the device (pointers into library memory).
struct LayerDev {
  const uint8_t* w_qkv;     // tiled dense [(Hq+2Hkv)hd][D], RoPE-paired rows
  const uint8_t* w_o;       // tiled dense [D][Hq hd]
  const uint8_t* w_pool;    // tiled dense [P][D]
  const uint8_t* w_router;  // tiled dense [E][P]
  const uint8_t* w_unpool;  // tiled dense [D][P]
  const uint16_t* attn_norm;  // bf16 [D]
  const uint16_t* moe_norm;   // bf16 [D]
  const float* router_bias;   // [E]
  const uint8_t* experts;     // [E][expert_bytes]
  const float* ts;            // [E][3] tensor scales gate, up, down
  int window;                 // 0 = global attention
  int loaded;
};

// Library scratch (device), sized at create time.
struct Scratch {
  uint16_t* q_stash;   // [T][Hq][hd] bf16, rotated queries of the next layer
  float* o_part;       // [nctas][64][hd] attention partial outputs
  float* ml_part;      // [nctas][64][2] running max / sum
  uint16_t* attn_o;    // [T][Hq hd]
  uint16_t* h1;        // [T][D]
  uint16_t* pooled;    // [T][P]
  uint16_t* a4;        // [T][P] f16: Q4(pooled) dequantised, the GEMM1 input
  float* logits;       // [T][E]
  uint8_t* sq_codes;   // [T k][I/2] fp4 intermediate
  uint8_t* sq_scales;  // [T k][I/16]
  uint16_t* y;         // [T k][P] expert outputs
  uint16_t* mvec;      // [T][P] combined expert output
  uint32_t* mc_cnt;    // [T][P/16] expert outputs in per (token, 16-row block); 0 between launches
  float* ss_part;      // [nctas][kMaxT] per-block sums of squares of the rows a residual projection wrote
  float* rope;         // [T][hd/2][2] cos, sin for the step's positions
  const double* inv_freq;  // [hd/2] theta^(-2i/d), a model constant
  unsigned long long* bar;  // grid barrier: arrivals since the last reset (a multiple of nctas between launches)
  uint32_t* err;       // [4] error word, phase, cta, spare
};

// The per-step part of a launch's arguments, kept in device memory for the
// captured step (a graph replays fixed kernel parameters; the positions and
// the tree change from step to step).  vis[0]: global layers, vis[1]:
// sliding-window layers.
struct StepInfo {
  int pos0;
  int depth[kMaxT];
  uint32_t vis[2][kMaxT];
};

struct LaunchArgs {
  Dims dm;
  LayerDev cur;
  LayerDev nxt;
  Scratch s;
  uint16_t* hidden;    // [T][D] in: h, out: h2
  uint16_t* kv_cur;    // [2][Hkv][max_seq][hd]
  uint16_t* kv_nxt;    // same for the next layer (unused when !has_next)
  const uint16_t* kv_nxt_ro;
  int pos0;             // cached length S: verify slot t's K/V row is S + t
  int depth[kMaxT];     // slot t's depth in the candidate tree: its position is pos0 + depth[t]
  uint32_t vis[kMaxT];  // verify slots slot t attends to (bit u): its ancestors and itself, inside the window
  int prologue;
  int has_next;
  const int* prev_routing;  // [T][topk] or null
  int* routing_out;         // [T][topk] or null
  unsigned long long budget_ns;
  unsigned long long* timeline;  // [nctas][kTimelineSlots] or null
  int inject_bar;
  int inject_cta;
  int kv_prefetch_rows;  // cap on next-layer KV rows prefetched into L2
  const StepInfo* step;  // device; when set, pos0 / depth / vis are read from it at launch start
};

// Host side: depth and attention masks of a candidate tree of T verify
// slots (parents[t] in [-1, t), -1 = a child of the last cached token;
// nullptr = the chain, parents[t] = t - 1) for a layer with the given
// window (0 = global): vis[t] has bit u set when slot u is an ancestor of
// t or t itself and its position lies in t's window.  Returns false if a
// parent is out of range.
inline bool tree_masks(const int32_t* parents, int T, int window, int* depth, uint32_t* vis) {
  uint32_t anc[kMaxT];
  for (int t = 0; t < T; ++t) {
    const int p = parents ? parents[t] : t - 1;
    if (p < -1 || p >= t) return false;
    depth[t] = p < 0 ? 0 : depth[p] + 1;
    anc[t] = (1u << t) | (p < 0 ? 0u : anc[p]);
  }
  for (int t = 0; t < T; ++t) {
    vis[t] = 0u;
    for (int u = 0; u < T; ++u)
      if (((anc[t] >> u) & 1u) && (window <= 0 || depth[u] > depth[t] - window)) vis[t] |= 1u << u;
  }
  for (int t = T; t < kMaxT; ++t) {
    depth[t] = 0;
    vis[t] = 0u;
  }
  return true;
}

}  // namespace msk
