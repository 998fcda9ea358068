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
//  NVFP4 expert e ("tiled expert", xexpert_bytes(P, I) bytes each): the
//  operand layout of the block-scaled tensor-core GEMMs, described below
//  (umma_code_off and the expert layout functions).
#pragma once

#include <cuda.h>

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
constexpr int kProducerWarp = kConsWarps;        // streams weights into shared memory
constexpr int kMmaWarp = kConsWarps + 1;         // issue the expert GEMMs' tensor-core operations: warps
constexpr int kMmaIssuers = 2;                   // kMmaWarp .. kMmaWarp + kMmaIssuers - 1, lane 0 each
constexpr int kThreads = kConsThreads + 32 * (1 + kMmaIssuers);  // + the producer and MMA warps
constexpr int kSlotBytes = 16384;                // weight ring slot
constexpr int kSlots = 5;                        // ring depth (80 KB)
constexpr int kMaxT = 16;                        // verify tokens
constexpr int kMaxK = 4096;                      // widest dense input
constexpr int kABytes = kMaxT * (kMaxK * 2 + 16);  // activation staging area (rows padded by 16 bytes)
constexpr int kAttnChunk = 64;                   // keys per KV stage (rows of one tiled copy)
constexpr int kAttnStages = 4;                   // KV stages (all but the one in use in flight)
constexpr int kTimelineSlots = 64;
// Timeline slots: [0, PH_COUNT) phase starts; 14 top-k chosen; 15 dispatch
// ready; 16 + phase: the block's work in a phase done; kSlotDense + 4 k +
// {0: entry (activations staged), 1: first weight tile in, 2: last group's
// products done} for the k-th dense projection of the launch; 30, 31: warp
// 0's logits loaded / top-k rounds done; 62, 63: attention's first KV chunk
// landed / key loop done.
constexpr int kSlotDense = 32;
// kSlotExpert + {0: GEMM1 token operands staged, 2: the block's GEMM1 work
// done (MMA issue or epilogue, whichever thread 0 ran), 3, 5: the same for
// GEMM2}
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
  PH_MCOMB,  // gated combine of the expert outputs
  PH_UNPOOL,
  PH_QKV,
  PH_END,
  PH_COUNT
};

MSK_HD inline constexpr size_t dense_tiled_bytes(int64_t N, int64_t K) { return (size_t)N * K * 2; }

// ---------------------------------------------------------------------------
// Operand layouts of the block-scaled tensor-core (tcgen05 kind::mxf4nvf4)
// expert GEMMs.  K-major, no swizzle: core matrices of 8 rows x 16 bytes
// (32 E2M1 elements, element 2i in the low nibble of byte i), the core
// matrix (kc, rg) of a [rows][K] operand at byte 128 (kc (rows / 8) + rg),
// so the descriptor offsets are LBO = 16 rows (along K) and SBO = 128
// (along rows).  One MMA (K = 64) reads core-matrix columns 2j, 2j + 1.
// Scale factors: per MMA a 512-byte chunk, row r = r32 + 32 r4 at byte
// 16 r32 + 4 r4 + b for its 16-element block b (0..3) of the MMA.
// ---------------------------------------------------------------------------
constexpr int kUStageK = 512;                 // K elements per weight stage (8 MMAs)
constexpr int kUStageBytes = 72 * kUStageK;   // 128 rows: 32 KB codes + 4 KB scale chunks
constexpr int kURows = 128;                   // MMA M (weight rows per unit)
constexpr int kUN = 16;                       // MMA N (token slots)

MSK_HD inline constexpr int umma_code_off(int rows, int r, int k) {
  return 128 * ((k >> 5) * (rows >> 3) + (r >> 3)) + 16 * (r & 7) + ((k & 31) >> 1);
}
MSK_HD inline constexpr int umma_sf_off(int r, int kblk) {
  return 512 * (kblk >> 2) + 16 * (r & 31) + 4 * (r >> 5) + (kblk & 3);
}
// K extent of stage s of a K-long unit (the last one may be 128).
MSK_HD inline constexpr int ustage_k(int K, int s) { return K - kUStageK * s < kUStageK ? K - kUStageK * s : kUStageK; }
// A weight stage of K extent kst: codes [0, 64 kst) in the layout above
// (rows = 128), then the scale chunks of its kst / 64 MMAs.
MSK_HD inline constexpr int ustage_bytes(int kst) { return 72 * kst; }
// Tiled expert e (xexpert_bytes each): GEMM1 units then GEMM2 units.  GEMM1
// unit b (I / 64 of them) is one M = 128 tile over K = P holding gate and up
// rows 64 b .. 64 b + 63 interleaved by 16: tile row 32 q + i is gate row
// 64 b + 16 q + i for i < 16 and up row 64 b + 16 q + i - 16 for i >= 16, so
// that each 32-lane quadrant of the accumulator holds matching gate and up
// rows.  GEMM2 unit b (P / 128 of them): down rows 128 b .. 128 b + 127 over
// K = I.  A unit is its stages in K order, stage s at kUStageBytes s.
MSK_HD inline constexpr size_t xg1_unit_bytes(int P) { return 72 * (size_t)P; }
MSK_HD inline constexpr size_t xg2_unit_bytes(int I) { return 72 * (size_t)I; }
MSK_HD inline constexpr size_t xg1_bytes(int P, int I) { return (size_t)(I / 64) * xg1_unit_bytes(P); }
MSK_HD inline constexpr size_t xexpert_bytes(int P, int I) { return xg1_bytes(P, I) + (size_t)(P / 128) * xg2_unit_bytes(I); }
// Byte offsets, within a tiled expert, of the code byte holding element k of
// row r of matrix `which` (0 gate, 1 up: [I][P]; 2 down: [P][I]) and of its
// block scale.
MSK_HD inline constexpr int xg1_tile_row(int which, int r) { return 32 * ((r & 63) >> 4) + 16 * which + (r & 15); }
MSK_HD inline constexpr size_t xcode_off(int P, int I, int which, int r, int k) {
  return which < 2 ? (size_t)(r >> 6) * xg1_unit_bytes(P) + (size_t)(k / kUStageK) * kUStageBytes +
                         umma_code_off(kURows, xg1_tile_row(which, r), k % kUStageK)
                   : xg1_bytes(P, I) + (size_t)(r >> 7) * xg2_unit_bytes(I) + (size_t)(k / kUStageK) * kUStageBytes +
                         umma_code_off(kURows, r & 127, k % kUStageK);
}
MSK_HD inline constexpr size_t xscale_off(int P, int I, int which, int r, int k) {
  return which < 2 ? (size_t)(r >> 6) * xg1_unit_bytes(P) + (size_t)(k / kUStageK) * kUStageBytes +
                         64 * ustage_k(P, k / kUStageK) + umma_sf_off(xg1_tile_row(which, r), (k % kUStageK) >> 4)
                   : xg1_bytes(P, I) + (size_t)(r >> 7) * xg2_unit_bytes(I) + (size_t)(k / kUStageK) * kUStageBytes +
                         64 * ustage_k(I, k / kUStageK) + umma_sf_off(r & 127, (k % kUStageK) >> 4);
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
  uint8_t* x4_codes;   // [T][P/2] Q4(pooled) E2M1 codes (element 2i in the low nibble of byte i): the GEMM1 input
  uint8_t* x4_scales;  // [T][P/16] its E4M3 block scales
  float* logits;       // [T][E]
  uint8_t* sq_codes;   // [T k][I/2] fp4 intermediate (same packing), the GEMM2 input
  uint8_t* sq_scales;  // [T k][I/16]
  uint16_t* y;         // [T k][P] expert outputs
  uint16_t* mvec;      // [T][P] combined expert output
  uint32_t* x1_done;   // [E] GEMM1 epilogue warps done per expert this launch; 0 between launches
  uint32_t* xq;        // [2 + E] GEMM2 work queue of the launch (0 between launches): [0] experts whose
                       // GEMM1 is complete, [1] GEMM2 units claimed, [2 + i] 1 + rank of the i-th such expert
  float* ss_part;      // [kMaxT][nctas] per-block sums of squares of the rows a residual projection wrote
  float* rope;         // [T][hd/2][2] cos, sin for the step's positions
  const double* inv_freq;  // [hd/2] theta^(-2i/d), a model constant
  unsigned long long* bar;  // grid barrier: arrivals since the last reset (a multiple of nctas between launches)
  uint32_t* err;       // [4] error word, phase, cta, spare
  int* pf_out;         // [1 + 32] block 0's ranked hot experts of the launch: count, then the experts
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
  int kv_z0;             // kv_map plane of this layer's K head 0 (its V heads follow the Hkv K heads)
  // The KV cache as a tiled-copy map: planes of [max_seq][hd] bf16 (one per
  // layer, K / V and kv head), boxes of 64 columns x kAttnChunk rows with
  // 128-byte swizzle.  Read by the copies from the kernel parameter itself.
  CUtensorMap kv_map;
};

// Encodes `map` for a KV cache of `planes` planes of [max_seq][hd] bf16 at
// `kv` (host; false if the driver rejects it).
bool encode_kv_map(CUtensorMap* map, const void* kv, int hd, int max_seq, long long planes);

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
