// Grouped GEMMs of the MoE expert layer on the sm_103a tensor cores.
//
// What they compute ("InternVL3.5 接入 pure FSDP2 后端开发实践", MindSpeed-MM
// issue 625, §2 fused expert layout gate_up_proj [E*H, 2I] / down_proj
// [E*I, H], §8.3 permute -> grouped_matmul -> SwiGLU -> grouped_matmul ->
// unpermute; "InternVL3.5 pure FSDP2 训练性能优化实践" §2.1: one grouped call
// over all experts instead of one call per expert):
//
//   FWD_GATEUP    h[r]      = silu(x[src_row[r]] . Wg_e) * (x[src_row[r]] . Wu_e)
//   FWD_DOWN      y_perm[r] = h[r] . Wd_e
//   DGRAD_DOWN    dgu[r]    = SwiGLU'(w[r] * (dy_perm[r] . Wd_e^T), gu_pre[r]), and
//                 the gate-weight gradient dw[r] = <dy_perm[r] . Wd_e^T, h[r]>
//                 (= <dY, y_perm[r]>) as per-tile partials, h recomputed in
//                 fp32 from the saved fp32 pre-activations
//   DGRAD_GATEUP  dx_perm[r]= dgu[r] . Wgu_e^T
//   WGRAD_DOWN    d_down_e  = (w h)_e^T . dy_perm_e
//   WGRAD_GATEUP  d_gu_e    = x[src_rows of e]^T . dgu_e
//   ROUTER        split-K partial router logits x . [W0; W1; W2] (see route.cu)
//
// One persistent, warp-specialised kernel template serves all of them (grid
// = the SM count, one CTA per SM).  A tile is 256 output columns by one or
// two 128-row halves (a per-mode choice, kH); the halves share each B tile:
// per 64-wide K block the CTA loads A (kH x 16 KB) and B (32 KB) and issues
// kH tcgen05.mma of M=128 x N=256.  Two halves need 7.6 KB of operands in
// shared memory per MFLOP instead of 11.4 KB, so the 192 KB ring (3 stages
// of 64 KB, or 4 of 48 KB with one half) hides more load latency.  Their two
// 128 x 256 fp32 accumulators fill the 512 TMEM columns, so the epilogue
// frees them as soon as it has read them into registers (packed to bf16),
// and stores after that while the next tile's MMAs run.  Modes whose
// epilogue cannot hold a tile row in registers (fp32 pre-activations saved
// for backward; the SwiGLU backward) use one half and double-buffered
// accumulators instead.  A tile whose rows end within its first half (the
// ragged tail of an expert) loads and multiplies only that half.
//   warp 0      TMA producer: A halves and B tiles into the ring, 128-byte
//               swizzled.  Gathered A rows (the permute fused into the load)
//               use cp.async.bulk.tensor ... tile::gather4, four token rows
//               per instruction.
//   warp 1      allocates the 512 TMEM columns and, from one lane, issues
//               tcgen05.mma (M=128, N=256, K=16, bf16 x bf16 -> fp32);
//               tcgen05.commit frees ring stages and hands finished
//               accumulators to the epilogue.
//   warps 2..9  epilogue: tcgen05.ld (one TMEM lane = one output row per
//               thread), fused SwiGLU / SwiGLU backward / gate weight in
//               fp32, vector stores.  With two halves warpgroup g drains half
//               g; with one half warpgroup g takes column half g.
//
// The tile list is derived on the device from expert_offsets (no host read
// back): forward and dgrad GEMMs are grouped along M (each expert's rows form
// ceil(M_e/BM) row tiles, empty experts none; gate_up, whose token rows a
// gather has just written, walks the experts from the last to the first, so
// that it starts on the rows still in L2); wgrad GEMMs are grouped along
// K (every expert owns a fixed grid of output tiles; its K extent is M_e,
// and an empty expert's tiles are written as zeros).  Within a wgrad tile,
// K rows past the expert's last row are zeroed in shared memory before the
// MMA so no other expert's rows leak in.  The K order inside a tile is fixed
// and there is no split-K with atomics: results are deterministic.
//
// Every spin wait is bounded (globaltimer); on expiry the kernel records
// MOE_ERR_TIMEOUT in the status word, lets the other roles stop, waits
// (bounded) for its TMA copies and MMAs in flight, frees its TMEM and
// returns.
#include "kernels.h"

namespace moe {

namespace {

constexpr int BMH = 128;                           // rows of one half (one MMA)
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int A_HALF_BYTES = BMH * BK * 2;         // 16 KB
constexpr int RING_BYTES = 192 * 1024;             // 3 x 64, 4 x 48 or 6 x 32 KB stages
constexpr int kEpiWarps = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MN_CHUNK_BYTES = 64 * 128;           // one 64-wide MN chunk x 64 K rows

enum Mode { FWD_GATEUP = 0, FWD_DOWN = 1, DGRAD_DOWN = 2, DGRAD_GATEUP = 3, WGRAD_DOWN = 4,
            WGRAD_GATEUP = 5, ROUTER = 6 };

// KH: 128-row halves per CTA (1 or 2); CG: CTAs per tile (1, or 2: a CTA
// pair issuing 2-SM MMAs, one 128-row half per CTA)
template <int MODE, int KH, int CG>
struct Traits {
  static constexpr bool kGateUp = (MODE == FWD_GATEUP);
  static constexpr bool kAMN = (MODE == WGRAD_DOWN || MODE == WGRAD_GATEUP);
  static constexpr bool kBMN = (kGateUp || MODE == FWD_DOWN || MODE == WGRAD_DOWN ||
                                MODE == WGRAD_GATEUP || MODE == ROUTER);
  static constexpr bool kKGrouped = (MODE == WGRAD_DOWN || MODE == WGRAD_GATEUP);
  // Tiles from the last expert to the first: when the permuted token rows
  // were written just before in increasing row order (moe_permute_rows, a
  // gather that moves more bytes than L2 holds), the rows of the last
  // experts are the ones still in L2.  Rows moved token by token
  // (moe_permute_rows_scatter) end in L2 in no expert order; either order
  // measures the same then.
  static constexpr bool kReverse = (MODE == FWD_GATEUP);
  static constexpr bool kRouter = (MODE == ROUTER);
  // One half per CTA for the epilogues with per-element math (SwiGLU, its
  // backward), which then overlap with the next tile's MMAs through two
  // accumulators, and for the router (few, narrow tiles: its K is split
  // instead); either for the plain bf16-store GEMMs.  A CTA pair holds one
  // half per CTA and half of each B tile, so a 256 x 256 tile moves 32 KB per
  // CTA per K block and keeps two accumulators.  The weight-gradient GEMMs
  // zero a tile's K rows past its expert in shared memory once the copies
  // have landed; in a pair rank 0's MMA warp zeroes both CTAs' stages (the
  // second CTA's through distributed shared memory).
  static_assert(KH == 1 || KH == 2, "one or two halves");
  static_assert(CG == 1 || CG == 2, "one CTA or a pair");
  static_assert(KH == 1 || (MODE != FWD_GATEUP && MODE != DGRAD_DOWN && MODE != ROUTER),
                "per-element epilogues use one half");
  static_assert(CG == 1 || (KH == 1 && MODE != ROUTER), "a pair holds one half per CTA; the router runs on single CTAs");
  static_assert(KH == 2 || CG == 2 || (MODE != WGRAD_DOWN && MODE != WGRAD_GATEUP),
                "wgrad uses 256-row tiles (two halves, or a pair)");
  static constexpr int kH = KH;
  static constexpr int kBM = kH * BMH * CG;          // rows of a tile
  static constexpr int kAccBufs = 2 / kH;
  // N of a tile: 256, or 128 for the router (E is often 128; split K gives
  // it its parallelism)
  static constexpr int kBN = (MODE == ROUTER) ? 128 : BN;
  static constexpr int kABytes = kH * A_HALF_BYTES;  // per CTA
  static constexpr int kBBytes = kBN * BK * 2 / CG;  // per CTA: a pair splits the N columns
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = RING_BYTES / kStageBytes;   // 4, 3, or 6 for a pair
  // read the accumulators into registers (bf16), free them, then store
  static constexpr bool kEarlyRelease = (kH == 2);
  // warp 0 TMA producer, warp 1 MMA issuer, then the epilogue warps
  static constexpr int kThreads = 32 * (2 + kEpiWarps);
};

struct GemmParams {   // 64-byte aligned through its CUtensorMap members
  CUtensorMap tmA;
  CUtensorMap tmB;
  const int32_t* offsets;   // [E+1] expert row offsets, or nullptr: one group of `rows`
  const int32_t* gidx;      // gather indices (src_row), or nullptr: identity
  const float* aux;         // fp32 gu_pre [R, 2I] read by DGRAD_DOWN
  const float* wrow;        // gate weight of each permuted row [R] (nullable)
  uint16_t* out;
  float* out_gu;            // FWD_GATEUP: fp32 pre-activations g | u [R, 2I] (nullable)
  uint16_t* out_hw;         // FWD_GATEUP: bf16(w_row * h) [R, I] (nullable, needs wrow)
  float* out_part;          // DGRAD_DOWN: per (row, 64-column block of I) partial of
                            // <dY . Wd^T, h> [R, I/64]; ROUTER: fp32 partial logits [parts, rows, n_out]
  uint32_t* status;
  uint64_t wait_limit_ns;
  int rows;                 // permuted rows R
  int E;
  int K;                    // contraction length (M-grouped modes; per part for ROUTER)
  int I;
  int n_out;                // valid output columns
  int m_w;                  // output rows per expert (K-grouped modes)
  int nt;                   // n tiles
  int mt_w;                 // m tiles per expert (K-grouped modes; per part for ROUTER)
  int64_t ldo;              // leading dimension of out
  int stall_producer;       // test hook: the producer issues no loads (a wait that runs out)
};

template <int MODE, int KH, int CG>
__device__ __forceinline__ uint32_t make_idesc(int m = BMH * CG) {
  using Tr = Traits<MODE, KH, CG>;
  return (1u << 4)                       // D: fp32
         | (1u << 7)                     // A: bf16
         | (1u << 10)                    // B: bf16
         | ((Tr::kAMN ? 1u : 0u) << 15)  // A major: 0 = K, 1 = MN
         | ((Tr::kBMN ? 1u : 0u) << 16)  // B major
         | ((uint32_t)(Tr::kBN >> 3) << 17)   // N
         | ((uint32_t)(m >> 4) << 24);   // M: one half, or 256 (128 for a half tile) over a pair
}

struct Tile {
  int e, mt, nt;
  int row0;       // M-grouped: first permuted row; K-grouped: first K row of the expert
  int rows;       // M-grouped: valid rows in the tile; K-grouped: K extent of the expert
  int kblocks;
  int halves;     // 128-row halves that carry valid output rows
  int half;       // a pair's tile of at most 128 rows: one M = 128 pair MMA, 64 rows per CTA
};

__device__ __forceinline__ void group_range(const GemmParams& p, int e, int& start, int& count) {
  if (p.offsets) {
    start = p.offsets[e];
    count = p.offsets[e + 1] - start;
  } else {
    start = 0;
    count = p.rows;
  }
}

template <int MODE, int KH, int CG>
__device__ __forceinline__ Tile decode_tile(const GemmParams& p, const int* prefix, int tile) {
  using Tr = Traits<MODE, KH, CG>;
  Tile t;
  t.half = 0;
  if (Tr::kRouter) {   // e = K part; rows of x in order; K range [e*K, (e+1)*K)
    const int per = p.mt_w * p.nt;
    t.e = tile / per;
    const int local = tile - t.e * per;
    t.mt = local / p.nt;
    t.nt = local - t.mt * p.nt;
    t.row0 = t.mt * Tr::kBM;
    t.rows = min(Tr::kBM, p.rows - t.row0);
    t.kblocks = p.K / BK;
    t.halves = t.rows > BMH ? 2 : 1;
  } else if (Tr::kKGrouped) {
    const int per = p.mt_w * p.nt;
    t.e = tile / per;
    const int local = tile - t.e * per;
    t.mt = local / p.nt;
    t.nt = local - t.mt * p.nt;
    group_range(p, t.e, t.row0, t.rows);
    t.kblocks = (t.rows + BK - 1) / BK;
    t.halves = (Tr::kBM == 2 * BMH && p.m_w - t.mt * Tr::kBM > BMH) ? 2 : 1;
  } else {
    if (Tr::kReverse) tile = prefix[p.E] - 1 - tile;
    int lo = 0, hi = p.E - 1;    // largest e with prefix[e] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    t.e = lo;
    const int local = tile - prefix[lo];
    t.mt = local / p.nt;
    t.nt = local - t.mt * p.nt;
    int start, count;
    group_range(p, t.e, start, count);
    t.row0 = start + t.mt * Tr::kBM;
    t.rows = min(Tr::kBM, count - t.mt * Tr::kBM);
    t.kblocks = p.K / BK;
    t.halves = (Tr::kBM == 2 * BMH && t.rows > BMH) ? 2 : 1;
    t.half = (CG == 2 && t.rows <= BMH) ? 1 : 0;
  }
  return t;
}

// Zero columns [c_lo, c_hi) of row m of an empty expert's weight-gradient
// tile (K-grouped modes).
__device__ __forceinline__ void store_zero_rows(const GemmParams& p, const Tile& t, int m, int c_lo,
                                               int c_hi) {
  if (m >= p.m_w) return;
  uint16_t* orow = p.out + ((int64_t)t.e * p.m_w + m) * p.ldo + (int64_t)t.nt * BN;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int c = c_lo; c < c_hi; c += 8)
    if (t.nt * BN + c < p.n_out) *reinterpret_cast<uint4*>(orow + c) = z;
}

// SwiGLU of the GEMM's fp32 gate and up values, h = silu(g) * u = g u / (1 + e^-g),
// with the fast exponential and division (relative error ~1e-6, far below the
// bf16 rounding of h).  An overflowing e^-g gives h = 0, the limit.  Every
// gate_up kernel uses it, so their results agree bit for bit.  The epilogue
// of a 128-column TMEM chunk (64 h columns, 128 rows, one warpgroup) measured
// about three times faster than with expf and a full division.
__device__ __forceinline__ float swiglu(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Transposes 16-byte chunks within each N-lane group of the warp (log2 N
// xor-butterfly stages of shuffles): on entry lane i holds chunks 0..N-1 of
// its own row in c[4j .. 4j+3]; on return it holds chunk (i % N) of the
// group's row j there.  The transpose is its own inverse.
template <int N>
__device__ __forceinline__ void transpose_chunks(uint32_t* c, int lane) {
#pragma unroll
  for (int b = 1; b < N; b <<= 1) {
    const bool hi = (lane & b) != 0;
#pragma unroll
    for (int pos = 0; pos < N; ++pos) {
      if (pos & b) continue;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t send = hi ? c[4 * pos + w] : c[4 * (pos | b) + w];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, b);
        if (hi) c[4 * pos + w] = recv;
        else c[4 * (pos | b) + w] = recv;
      }
    }
  }
}

// Stores a block of 32 rows x 16N bytes (N = 8: 128, N = 4: 64) held one
// row per lane (c: that row's bytes).  After the transpose every store
// instruction writes 32/N whole row segments, where one row per lane would
// touch 32 lines per instruction and write each 32-byte sector in two halves.
// base: the block's first byte in the warp's row 0; ld: row pitch in bytes;
// rows whose bit is clear in row_mask are skipped.  Warp-wide.
template <int N>
__device__ __forceinline__ void store_block(uint8_t* base, int64_t ld, uint32_t* c, int lane,
                                            uint32_t row_mask) {
  transpose_chunks<N>(c, lane);
  const int g = lane / N, i = lane % N;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const int row = N * g + j;
    if ((row_mask >> row) & 1u)
      *reinterpret_cast<uint4*>(base + row * ld + 16 * i) =
          make_uint4(c[4 * j], c[4 * j + 1], c[4 * j + 2], c[4 * j + 3]);
  }
}

__device__ __forceinline__ void store_block128(uint8_t* base, int64_t ld, uint32_t* c, int lane,
                                               uint32_t row_mask) {
  store_block<8>(base, ld, c, lane, row_mask);
}

// The inverse of store_block<8>: reads 32 rows x 128 bytes with four whole
// rows per load instruction, then transposes so that lane l holds row l's
// 128 bytes in c.  Rows whose bit is clear in row_mask read as zeros.
__device__ __forceinline__ void load_block128(const uint8_t* base, int64_t ld, uint32_t* c, int lane,
                                              uint32_t row_mask) {
  const int g = lane >> 3, i = lane & 7;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int row = 8 * g + j;
    uint4 q = make_uint4(0, 0, 0, 0);
    if ((row_mask >> row) & 1u) q = __ldg(reinterpret_cast<const uint4*>(base + row * ld + 16 * i));
    c[4 * j] = q.x; c[4 * j + 1] = q.y; c[4 * j + 2] = q.z; c[4 * j + 3] = q.w;
  }
  transpose_chunks<8>(c, lane);
}

// The copies of one K block of a tile: A (KH halves or MN chunks) and B into
// the stage at sA / sB, completing on the barrier fb.  In a CTA pair, CTA
// `crank` copies its own 128 rows of A and its half of the B columns (chunks
// 2 crank, 2 crank + 1 of the tile's four 64-wide chunks) into its own
// stage; the bytes of both count on rank 0's barrier.
// Warp-wide: gathered loads spread over the lanes, the others are issued by
// lane 0.
template <int MODE, int KH, int CG>
__device__ __forceinline__ void stage_loads(const GemmParams& p, const Tile& t, int kb, uint32_t sA,
                                            uint32_t sB, uint32_t fb, int lane, int crank,
                                            const int (&gi)[KH][4], uint64_t keep_x) {
  using Tr = Traits<MODE, KH, CG>;
  // a pair's copies count on rank 0's barrier (fb is its shared::cluster address)
  auto tma_load_2d = [&](uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    if (CG == 2) tma_load_2d_pair(dst, map, x, y, bar);
    else ::moe::tma_load_2d(dst, map, x, y, bar);
  };
  auto tma_gather4_hint = [&](uint32_t dst, const CUtensorMap* map, int x, int r0, int r1, int r2, int r3,
                              uint32_t bar, uint64_t pol) {
    if (CG == 2) tma_gather4_pair_hint(dst, map, x, r0, r1, r2, r3, bar, pol);
    else ::moe::tma_gather4_hint(dst, map, x, r0, r1, r2, r3, bar, pol);
  };
  const int k0 = kb * BK;
  const int ah = CG == 2 ? 1 : t.halves;             // A halves this CTA loads
  // M-grouped: its first A row (a pair's half tile: 64 rows per CTA, of which
  // the 128-row box brings the first 64 into use)
  const int arow0 = t.row0 + crank * (t.half ? BMH / 2 : BMH);
  const int c0 = CG == 2 ? 2 * crank : 0;            // its first B chunk of the tile
  const int nc = CG == 2 ? 2 : 4;
  if (Tr::kGateUp) {
    if (p.gidx) {                                    // permute fused into the load (TMA)
      for (int h = 0; h < ah; ++h)
        tma_gather4_hint(sA + h * A_HALF_BYTES + 4 * lane * 128, &p.tmA, k0, gi[h][0], gi[h][1],
                         gi[h][2], gi[h][3], fb, keep_x);
    } else if (lane == 0) {                          // rows already in permuted order
      for (int h = 0; h < ah; ++h)
        tma_load_2d(sA + h * A_HALF_BYTES, &p.tmA, k0, arow0 + h * BMH, fb);
    }
    if (lane == 0) {
      const int brow = t.e * p.K + k0;               // gate_up rows of expert e
      const int n0 = t.nt * 128;                     // chunks: gate n0, n0+64; up I+n0, I+n0+64
      for (int c = 0; c < nc; ++c) {
        // a pair's half tile folds each CTA's 256 columns into two TMEM lane
        // halves of 128: CTA r takes gate and up chunk r, so that a row's
        // gate and up columns share a TMEM lane
        const int cc = (CG == 2 && t.half) ? (c == 0 ? crank : 2 + crank) : c0 + c;
        tma_load_2d(sB + c * MN_CHUNK_BYTES, &p.tmB, (cc >> 1) * p.I + n0 + 64 * (cc & 1), brow, fb);
      }
    }
  } else if (MODE == ROUTER) {
    if (lane == 0) {
      const int kg = t.e * p.K + k0;                 // row of the stacked [W0; W1; W2]
      for (int h = 0; h < t.halves; ++h)             // x repeats along the stacked K
        tma_load_2d(sA + h * A_HALF_BYTES, &p.tmA, kg % p.I, t.row0 + h * BMH, fb);
      const int n0 = t.nt * Tr::kBN;
#pragma unroll
      for (int c = 0; c < Tr::kBN / 64; ++c) tma_load_2d(sB + c * MN_CHUNK_BYTES, &p.tmB, n0 + 64 * c, kg, fb);
    }
  } else if (MODE == FWD_DOWN) {
    if (lane == 0) {
      for (int h = 0; h < ah; ++h)
        tma_load_2d(sA + h * A_HALF_BYTES, &p.tmA, k0, arow0 + h * BMH, fb);
      const int brow = t.e * p.K + k0;               // down rows of expert e
      const int n0 = t.nt * BN;
      for (int c = 0; c < nc; ++c)
        tma_load_2d(sB + c * MN_CHUNK_BYTES, &p.tmB, n0 + 64 * (c0 + c), brow, fb);
    }
  } else if (MODE == DGRAD_DOWN || MODE == DGRAD_GATEUP) {
    if (lane == 0) {
      for (int h = 0; h < ah; ++h)
        tma_load_2d(sA + h * A_HALF_BYTES, &p.tmA, k0, arow0 + h * BMH, fb);
      // B^T rows: expert e's block of rows_per_e rows, K-major (one box of
      // BN / CG rows)
      const int rows_per_e = (MODE == DGRAD_DOWN) ? p.I : p.n_out;
      tma_load_2d(sB, &p.tmB, k0, t.e * rows_per_e + t.nt * BN + crank * (BN / 2), fb);
    }
  } else {  // WGRAD_*: A = rows of the expert (K = tokens), MN-major chunks of 64 m
    const int krow = t.row0 + k0;
    const int m0 = t.mt * Tr::kBM + crank * BMH;
    const int ac = CG == 2 ? 2 : 2 * t.halves;      // A chunks this CTA loads
    if (MODE == WGRAD_GATEUP && p.gidx) {            // gathered through src_row
      // lane: MN chunk c = lane >> 3, K rows 8*(lane & 7) .. +7 (two gather4)
      const int c = lane >> 3;
      if (c < ac) {
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const int kr0 = 8 * (lane & 7) + 4 * q2;
          int r4[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) r4[q] = p.gidx[t.row0 + min(k0 + kr0 + q, t.rows - 1)];
          tma_gather4_hint(sA + c * MN_CHUNK_BYTES + kr0 * 128, &p.tmA, m0 + 64 * c, r4[0], r4[1],
                           r4[2], r4[3], fb, keep_x);
        }
      }
    } else if (lane == 0) {                          // rows already in permuted order
      for (int c = 0; c < ac; ++c)
        tma_load_2d(sA + c * MN_CHUNK_BYTES, &p.tmA, m0 + 64 * c, krow, fb);
    }
    if (lane == 0) {
      const int n0 = t.nt * BN;
      for (int c = 0; c < nc; ++c)
        tma_load_2d(sB + c * MN_CHUNK_BYTES, &p.tmB, n0 + 64 * (c0 + c), krow, fb);
    }
  }
}

// Zeroes the K rows [kvalid, 64) of every 64 x 128-byte chunk of a stage (a
// weight-gradient tile's last K block may run past its expert's rows).  Lane
// l writes 16-byte unit l % 8 of rows kvalid + l / 8, +4, ... of each chunk:
// no divisions on the MMA issuer's path.  Warp-wide; makes the writes
// visible to the tensor cores.
template <int STAGE_BYTES>
__device__ __forceinline__ void zero_k_tail(uint8_t* stage, int kvalid, int lane) {
  constexpr int kChunks = STAGE_BYTES / MN_CHUNK_BYTES;
  uint8_t* unit = stage + (lane & 7) * 16;
#pragma unroll
  for (int chunk = 0; chunk < kChunks; ++chunk)
    for (int row = kvalid + (lane >> 3); row < BK; row += 4)
      *reinterpret_cast<uint4*>(unit + chunk * MN_CHUNK_BYTES + row * 128) = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncwarp();
}

// The same for a CTA pair, from rank 0's MMA warp once both CTAs' copies of
// the stage have landed: its own stage, and the second CTA's (same offset in
// that CTA's shared memory) through distributed shared memory.  The writes
// are made visible at cluster scope and to the tensor cores' async proxy
// before the pair MMA that reads both stages is issued.
template <int STAGE_BYTES>
__device__ __forceinline__ void zero_k_tail_pair(uint8_t* stage, int kvalid, int lane) {
  constexpr int kChunks = STAGE_BYTES / MN_CHUNK_BYTES;
  uint8_t* unit = stage + (lane & 7) * 16;
  const uint32_t peer = mapa_shared(smem_u32(unit), 1);
#pragma unroll
  for (int chunk = 0; chunk < kChunks; ++chunk)
    for (int row = kvalid + (lane >> 3); row < BK; row += 4) {
      const int off = chunk * MN_CHUNK_BYTES + row * 128;
      *reinterpret_cast<uint4*>(unit + off) = make_uint4(0, 0, 0, 0);
      st_shared_cluster_zero16(peer + (uint32_t)off);
    }
  fence_acq_rel_cluster();
  fence_proxy_async_all();
  __syncwarp();
}

template <int MODE, int KH, int CG>
__global__ void __launch_bounds__(Traits<MODE, KH, CG>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
  using Tr = Traits<MODE, KH, CG>;
  constexpr int STAGES = Tr::kStages;
  constexpr bool kPair = (CG == 2);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RING_BYTES);
  // bars: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain (at most 17 of 24)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 24);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* prefix = reinterpret_cast<int*>(tmem_slot + 2);   // [E+1], then the offsets check flag

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // In a CTA pair: rank 0 issues the MMAs for both; each CTA loads its own
  // operand halves into its own ring and drains its own 128 TMEM lanes.
  const int crank = kPair ? (int)cluster_ctarank() : 0;
  const int tile0 = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int tile_step = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const uint32_t ring_u32 = smem_u32(ring);
  const uint32_t bar_u32 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar_u32 + 8u * s; };
  auto empty_bar = [&](int s) { return bar_u32 + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bar_u32 + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar_u32 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar_u32 + 8u * (2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // in a pair only rank 0's full barriers are used: its producer arrives
      // and expects the bytes of both CTAs
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kEpiWarps * CG);   // one arrive per epilogue warp (of both CTAs)
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
  }
  if (warp == 1) {
    if (kPair) {
      tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  pdl_wait();      // the set-up above overlaps the kernel before this one
  pdl_trigger();
  // Tile prefix over experts (M-grouped modes): prefix[e] = sum_{e'<e} ceil(M_e'/BM) * nt.
  // Tiles go out in expert order, so the row tiles of one expert run at about
  // the same time and read its weights from L2 after the first of them.
  // Expert offsets that are not an exclusive scan of counts ending at the row
  // count (offsets[0] = 0, non-decreasing, offsets[E] = rows) are reported
  // and the launch does no work: no tile may store past its output or run
  // for an unbounded K.
  int total_tiles;
  if (warp == 2) {
    bool bad = false;
    if (p.offsets && !Tr::kRouter) {
      for (int e0 = 0; e0 <= p.E; e0 += 32) {
        const int e = e0 + lane;
        if (e <= p.E) {
          const int v = p.offsets[e];
          const int prev = e > 0 ? p.offsets[e - 1] : 0;
          if (v < prev || v > p.rows || (e == 0 && v != 0) || (e == p.E && v != p.rows)) bad = true;
        }
      }
      bad = __any_sync(0xffffffffu, bad);
      if (bad && lane == 0) report_status(p.status, kStatusDevice, kKernGemm, 5);
    }
    if (lane == 0) prefix[p.E + 1] = bad ? 1 : 0;
  }
  if (Tr::kKGrouped || Tr::kRouter) {
    total_tiles = p.E * p.mt_w * p.nt;
  } else {
    if (warp == 2) {
      const bool bad = __shfl_sync(0xffffffffu, lane == 0 ? prefix[p.E + 1] : 0, 0) != 0;
      int carry = 0;
      for (int e0 = 0; e0 < p.E; e0 += 32) {
        const int e = e0 + lane;
        int v = 0;
        if (e < p.E && !bad) {
          int start, count;
          group_range(p, e, start, count);
          v = ((count + Tr::kBM - 1) / Tr::kBM) * p.nt;
        }
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += n;
        }
        if (e < p.E) prefix[e] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) prefix[p.E] = carry;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync_all();   // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (!Tr::kKGrouped && !Tr::kRouter) total_tiles = prefix[p.E];
  if (prefix[p.E + 1]) total_tiles = 0;   // invalid expert offsets (reported above)

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    // Gathered token rows are re-read by every expert a token was routed to,
    // spread over the whole launch while the weights stream through L2: keep
    // them resident.
    const uint64_t keep_x = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0;       // stages that ever received a load
    uint32_t last_parity = 0;       // bit s: parity of the last load into stage s
    bool ok = true;
    for (int tile = tile0; tile < total_tiles && ok && !p.stall_producer; tile += tile_step) {
      const Tile t = decode_tile<MODE, KH, CG>(p, prefix, tile);
      if (t.kblocks == 0) continue;
      int gi[Tr::kH][4];
      if (Tr::kGateUp && p.gidx) {   // lane's rows: 4*lane .. +3 of each of this CTA's halves
#pragma unroll
        for (int h = 0; h < Tr::kH; ++h)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            gi[h][q] = p.gidx[t.row0 + min(crank * (t.half ? BMH / 2 : BMH) + h * BMH + 4 * lane + q, t.rows - 1)];
      }
      const uint32_t a_bytes = (uint32_t)((kPair ? 1 : t.halves) * A_HALF_BYTES);
      for (int kb = 0; kb < t.kblocks; ++kb) {
        ok = mbar_wait_warp<kPair>(empty_bar(stage), phase ^ 1u, abort_flag, p.wait_limit_ns, p.status, 1);
        if (!ok) break;
        const uint32_t sA = ring_u32 + stage * Tr::kStageBytes;
        const uint32_t sB = sA + Tr::kABytes;
        const uint32_t fb = (kPair && crank != 0) ? mapa_shared(full_bar(stage), 0) : full_bar(stage);
        if (lane == 0 && crank == 0)
          mbar_arrive_expect_tx(fb, (uint32_t)CG * (a_bytes + (uint32_t)Tr::kBBytes));
        __syncwarp();
        stage_loads<MODE, KH, CG>(p, t, kb, sA, sB, fb, lane, crank, gi, keep_x);
        issued_mask |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0 && crank == 0) {
      // stopped early: wait (bounded) for the copies still in flight (in a
      // pair rank 0's barriers count both CTAs' copies)
      for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s)) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(full_bar(s), (last_parity >> s) & 1u) &&
                 globaltimer_ns() - t0 < p.wait_limit_ns) {
          }
        }
    }
  } else if (warp == 1 && crank != 0) {
    // the second CTA of a pair issues no MMAs: rank 0 issues them for both
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    const uint32_t idesc = make_idesc<MODE, KH, CG>();
    const uint32_t idesc_half = make_idesc<MODE, KH, CG>(BMH);   // a pair's half tile
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;                 // accumulator buffer (always 0 with two halves)
    uint32_t acc_phase = 0;
    bool ok = true;
    bool issued_any = false;
    for (int tile = tile0; tile < total_tiles && ok; tile += tile_step) {
      const Tile t = decode_tile<MODE, KH, CG>(p, prefix, tile);
      if (t.kblocks == 0) continue;
      // the epilogue (of both CTAs) has drained this accumulator buffer
      ok = mbar_wait_warp<kPair>(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.wait_limit_ns, p.status, 2);
      if (!ok) break;
      tc_fence_after();
      for (int kb = 0; kb < t.kblocks; ++kb) {
        ok = mbar_wait_warp<kPair>(full_bar(stage), phase, abort_flag, p.wait_limit_ns, p.status, 3);
        if (!ok) break;
        const uint32_t sA = ring_u32 + stage * Tr::kStageBytes;
        const uint32_t sB = sA + Tr::kABytes;
        if (Tr::kKGrouped && t.rows - kb * BK < BK) {   // K rows past the expert's last row
          if (kPair) zero_k_tail_pair<Tr::kStageBytes>(ring + stage * Tr::kStageBytes, t.rows - kb * BK, lane);
          else zero_k_tail<Tr::kStageBytes>(ring + stage * Tr::kStageBytes, t.rows - kb * BK, lane);
        }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = Tr::kBMN ? umma_desc(sB + kk * 2048, MN_CHUNK_BYTES, 1024)
                                         : umma_desc(sB + kk * 32, 16, 1024);
            if (kPair) {   // one M = 256 MMA over both CTAs' halves
              const uint64_t ad = Tr::kAMN ? umma_desc(sA + kk * 2048, MN_CHUNK_BYTES, 1024)
                                           : umma_desc(sA + kk * 32, 16, 1024);
              tc_mma_bf16_pair(tmem_base + (uint32_t)(acc * BN), ad, bd, t.half ? idesc_half : idesc,
                               (kb | kk) != 0 ? 1u : 0u);
            } else {
              for (int h = 0; h < t.halves; ++h) {
                const uint32_t aBase = sA + h * A_HALF_BYTES;
                const uint64_t ad = Tr::kAMN ? umma_desc(aBase + kk * 2048, MN_CHUNK_BYTES, 1024)
                                             : umma_desc(aBase + kk * 32, 16, 1024);
                tc_mma_bf16(tmem_base + (uint32_t)((acc + h) * BN), ad, bd, idesc,
                            (kb | kk) != 0 ? 1u : 0u);
              }
            }
          }
          if (kPair) tc_commit_pair(empty_bar(stage), 3);   // frees the stage in both CTAs
          else tc_commit(empty_bar(stage));
        }
        issued_any = true;
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) {
        if (kPair) tc_commit_pair(accf_bar(acc), 3);
        else tc_commit(accf_bar(acc));
      }
      __syncwarp();
      if (++acc == Tr::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && issued_any && lane == 0) {
      // stopped early: make sure every MMA issued has finished before TMEM is freed
      if (kPair) tc_commit_pair(drain_bar, 1);
      else tc_commit(drain_bar);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain_bar, 0) && globaltimer_ns() - t0 < p.wait_limit_ns) {
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    // Each warp reads the TMEM lane quarter its rank allows (warp % 4).  With
    // two halves warpgroup wg drains half wg (all 256 columns); with one,
    // warpgroup wg takes columns [128 wg, 128 wg + 128) of the single half
    // (in a pair: of this CTA's 128 rows of the 256-row tile).
    const int quarter = warp & 3;                     // TMEM lanes 32*quarter .. +31
    const int wg = (warp - 2) >> 2;
    const int half = Tr::kH == 2 ? wg : 0;
    const int rbase = crank * BMH;                    // this CTA's first row of the tile
    const int r = rbase + half * BMH + quarter * 32 + lane;   // tile row of this thread
    // a warp's arrive that frees an accumulator buffer (rank 0's barrier in a pair)
    auto release = [&](uint32_t bar) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair && crank != 0) mbar_arrive_cluster(mapa_shared(bar, 0));
        else mbar_arrive(bar);
      }
    };
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = tile0; tile < total_tiles; tile += tile_step) {
      const Tile t = decode_tile<MODE, KH, CG>(p, prefix, tile);
      if (t.kblocks == 0) {
        if (Tr::kKGrouped) {   // an empty expert: zero its weight-gradient tile
          if (Tr::kH == 2) store_zero_rows(p, t, t.mt * Tr::kBM + r, 0, BN);
          else store_zero_rows(p, t, t.mt * Tr::kBM + r, 128 * wg, 128 * wg + 128);
        }
        continue;
      }
      // every lane acquires the accumulator itself before the warp reads it
      if (!mbar_wait_warp<kPair>(accf_bar(acc), acc_phase, abort_flag, p.wait_limit_ns, p.status, 4)) break;
      tc_fence_after();
      const bool active = half < t.halves;     // warp-uniform
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)((acc + half) * BN);
      const uint32_t done = acce_bar(acc);
      if (++acc == Tr::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
      // Rows of this warp: 32 consecutive tile rows starting at wrow (one
      // per lane); stores go through store_block (whole row segments).  A
      // pair's half tile folds each CTA's 64 rows x 256 columns into TMEM
      // lanes: lane L holds row 64 r + L % 64, columns 128 (L / 64) .. +127
      // in TMEM columns 0..127 (nh = L / 64 for this warp).
      const bool ht = kPair && t.half;   // warp-uniform
      const int nh = quarter >> 1;
      const int wrow = ht ? crank * (BMH / 2) + 32 * (quarter & 1) : rbase + half * BMH + quarter * 32;
      float v[32];
      if (Tr::kEarlyRelease) {
        // read the whole row into registers as bf16 (16 columns at a time:
        // the packed row already takes 128 registers), free the accumulator,
        // then store while the next tile's MMAs run
        uint32_t pk[BN / 2];
        if (active) {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            tmem_ld16(taddr + 16 * c, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) pk[8 * c + q] = pack_bf16x2(v[2 * q], v[2 * q + 1]);
          }
        }
        release(done);
        if (active) {
          uint8_t* base;
          uint32_t row_mask;
          const int n0 = t.nt * BN;
          if (Tr::kKGrouped) {   // rows m = mt*BM + r of expert e's weight-gradient block
            const int m0 = t.mt * Tr::kBM + wrow;
            row_mask = __ballot_sync(0xffffffffu, m0 + lane < p.m_w);
            base = reinterpret_cast<uint8_t*>(p.out + ((int64_t)t.e * p.m_w + m0) * p.ldo + n0);
          } else {
            row_mask = __ballot_sync(0xffffffffu, wrow + lane < t.rows);
            base = reinterpret_cast<uint8_t*>(p.out + (int64_t)(t.row0 + wrow) * p.ldo + n0);
          }
#pragma unroll
          for (int blk = 0; blk < BN / 64; ++blk)
            if (n0 + 64 * blk < p.n_out)
              store_block128(base + 128 * blk, p.ldo * 2, pk + 32 * blk, lane, row_mask);
        }
        continue;
      }
      if (!active) {
        // this half carries no rows of the tile: nothing to read or store
      } else if (MODE == FWD_GATEUP) {
        // warpgroup wg: h columns [64 wg, 64 wg + 64) of the tile (gate and
        // up accumulator columns c and 128 + c); in a pair's half tile h
        // columns 64 nh + [32 wg, 32 wg + 32) (gate at TMEM column c, up at
        // 64 + c)
        const uint32_t row_mask = __ballot_sync(0xffffffffu, wrow + lane < t.rows);
        const int64_t row0 = t.row0 + wrow;
        {
          const bool row_ok = wrow + lane < t.rows;
          const float wr = (p.out_hw && row_ok) ? p.wrow[row0 + lane] : 0.f;
#pragma unroll 1
          for (int c = 0; c < (ht ? 1 : 2); ++c) {         // 32 h columns at a time
            const int gcol = ht ? 32 * wg : 64 * wg + 32 * c;            // TMEM column of the gate values
            const int ucol = ht ? 64 + 32 * wg : 128 + 64 * wg + 32 * c;  // ... of the up values
            const int col = t.nt * 128 + (ht ? 64 * nh + 32 * wg : 64 * wg + 32 * c);   // h column
            if (col >= p.n_out) break;                     // warp-uniform
            uint32_t bits[32];
            if (p.out_gu) {                                // fp32 pre-activations g | u, 128-byte blocks
#pragma unroll
              for (int gu = 0; gu < 2; ++gu) {
                tmem_ld32(taddr + (gu ? ucol : gcol), v);
#pragma unroll
                for (int q = 0; q < 32; ++q) bits[q] = __float_as_uint(v[q]);
                store_block128(reinterpret_cast<uint8_t*>(p.out_gu + row0 * 2 * p.I + gu * p.I + col), 8 * p.I,
                               bits, lane, row_mask);
              }
            }
            float u[32];
            tmem_ld32(taddr + gcol, v);                    // gate columns
            tmem_ld32(taddr + ucol, u);                    // up columns
            // bits[0..15]: h, bits[16..31]: w * h (bf16 pairs)
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float h0 = swiglu(v[2 * q], u[2 * q]), h1 = swiglu(v[2 * q + 1], u[2 * q + 1]);
              bits[q] = pack_bf16x2(h0, h1);
              bits[16 + q] = pack_bf16x2(h0 * wr, h1 * wr);
            }
            store_block<4>(reinterpret_cast<uint8_t*>(p.out + row0 * p.ldo + col), p.ldo * 2, bits, lane,
                           row_mask);
            if (p.out_hw)   // warp-uniform
              store_block<4>(reinterpret_cast<uint8_t*>(p.out_hw + row0 * p.ldo + col), p.ldo * 2, bits + 16,
                             lane, row_mask);
          }
        }
      } else if (MODE == ROUTER) {   // fp32 partial logits; warpgroup wg: columns [64 wg, 64 wg + 64)
        const bool row_ok = wrow + lane < t.rows;
        const uint32_t row_mask = __ballot_sync(0xffffffffu, row_ok);
        float* orow0 = p.out_part + ((int64_t)t.e * p.rows + t.row0 + wrow) * p.ldo;
        const int n0 = t.nt * Tr::kBN;
#pragma unroll 1
        for (int c0 = (Tr::kBN / 2) * wg; c0 < (Tr::kBN / 2) * (wg + 1); c0 += 32) {
          if (n0 + c0 >= p.n_out) break;                 // warp-uniform
          tmem_ld32(taddr + c0, v);
          if (n0 + c0 + 32 <= p.n_out && (p.ldo & 3) == 0) {   // whole 128-byte row segments
            uint32_t bits[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) bits[q] = __float_as_uint(v[q]);
            store_block128(reinterpret_cast<uint8_t*>(orow0 + n0 + c0), p.ldo * 4, bits, lane, row_mask);
          } else if (row_ok) {
            float* orow = orow0 + (int64_t)lane * p.ldo;
#pragma unroll
            for (int q = 0; q < 32; ++q)
              if (n0 + c0 + q < p.n_out) orow[n0 + c0 + q] = v[q];
          }
        }
      } else if (MODE == FWD_DOWN || MODE == DGRAD_GATEUP || Tr::kKGrouped) {   // one half: column half wg
        // (a pair's half tile: columns 128 nh + [64 wg, 64 wg + 64), one block)
        const int n0 = t.nt * BN + (ht ? 128 * nh + 64 * wg : 128 * wg);
        const int tc0 = ht ? 64 * wg : 128 * wg;         // TMEM column of the first block
        uint32_t row_mask;
        uint8_t* base;
        if (Tr::kKGrouped) {   // rows m = mt*BM + r of expert e's weight-gradient block
          const int m0 = t.mt * Tr::kBM + wrow;
          row_mask = __ballot_sync(0xffffffffu, m0 + lane < p.m_w);
          base = reinterpret_cast<uint8_t*>(p.out + ((int64_t)t.e * p.m_w + m0) * p.ldo + n0);
        } else {
          row_mask = __ballot_sync(0xffffffffu, wrow + lane < t.rows);
          base = reinterpret_cast<uint8_t*>(p.out + (int64_t)(t.row0 + wrow) * p.ldo + n0);
        }
#pragma unroll 1
        for (int blk = 0; blk < (ht ? 1 : 2); ++blk) {
          if (n0 + 64 * blk >= p.n_out) break;
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            tmem_ld32(taddr + tc0 + 64 * blk + 32 * c, v);
#pragma unroll
            for (int q = 0; q < 16; ++q) pk[16 * c + q] = pack_bf16x2(v[2 * q], v[2 * q + 1]);
          }
          store_block128(base + 128 * blk, p.ldo * 2, pk, lane, row_mask);
        }
      } else if (MODE == DGRAD_DOWN) {
        const bool row_ok = wrow + lane < t.rows;
        const uint32_t row_mask = __ballot_sync(0xffffffffu, row_ok);
        const int64_t row = t.row0 + wrow + lane;
        const int64_t row0 = t.row0 + wrow;
        // columns as in the bf16 path: 128 wg + [0, 128), or in a pair's half
        // tile 128 nh + 64 wg + [0, 64)
        const int n0 = t.nt * BN + (ht ? 128 * nh + 64 * wg : 128 * wg);
        const int tc0 = ht ? 64 * wg : 128 * wg;
        const int nparts = (p.n_out + 63) / 64;          // one dw partial per 64 columns
        const float wr = row_ok ? p.wrow[row] : 0.f;     // dh = w * (dY . Wd^T)
        float dot = 0.f;                                 // <dY . Wd^T, h> over a 64-column block
        const uint8_t* aux0 = reinterpret_cast<const uint8_t*>(p.aux + row0 * 2 * p.I);
        uint8_t* out0 = reinterpret_cast<uint8_t*>(p.out + row0 * 2 * p.I);
#pragma unroll 1
        for (int c = 0; c < (ht ? 2 : 4); ++c) {         // 32 columns at a time
          const int col = n0 + 32 * c;
          if (col >= p.n_out) break;                     // blocks of 64 are whole (I % 64 == 0)
          tmem_ld32(taddr + tc0 + 32 * c, v);            // dY . Wd^T (fp32)
          uint32_t gb[32], ub[32];                       // the row's fp32 pre-activations g | u
          load_block128(aux0 + 4 * col, 8 * p.I, gb, lane, row_mask);
          load_block128(aux0 + 4 * (p.I + col), 8 * p.I, ub, lane, row_mask);
          uint32_t dg[16], du[16];
#pragma unroll
          for (int q = 0; q < 32; q += 2) {
            float o[2][2];
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const float g = __uint_as_float(gb[q + e2]), u = __uint_as_float(ub[q + e2]);
              const float s = 1.0f / (1.0f + expf(-g));
              dot = fmaf(v[q + e2], g * s * u, dot);     // h = silu(g) * u from the fp32 pre-activations
              const float dh = wr * v[q + e2];
              o[0][e2] = dh * u * s * (1.0f + g * (1.0f - s));
              o[1][e2] = dh * g * s;
            }
            dg[q / 2] = pack_bf16x2(o[0][0], o[0][1]);
            du[q / 2] = pack_bf16x2(o[1][0], o[1][1]);
          }
          store_block<4>(out0 + 2 * col, 4 * p.I, dg, lane, row_mask);
          store_block<4>(out0 + 2 * (p.I + col), 4 * p.I, du, lane, row_mask);
          if (c & 1) {                                   // a 64-column block is done
            if (row_ok && p.out_part) p.out_part[row * nparts + col / 64] = dot;
            dot = 0.f;
          }
        }
      }
      release(done);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync_all();   // neither CTA frees TMEM or leaves while the other may signal it
  if (warp == 1) {
    tc_fence_after();
    if (kPair) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ring, 24 mbarriers, TMEM slot + abort flag, prefix[E + 1] + the offsets check flag, slack
size_t gemm_smem_bytes(int E) { return 1024 + (size_t)RING_BYTES + 8 * 24 + 16 + 4 * (size_t)(E + 2) + 64; }

// Persistent launch: one CTA per SM, or one pair per two SMs (a cluster of
// two CTAs; as many clusters as fit at once, capped by the tile count).
template <int MODE, int KH, int CG>
cudaError_t run_gemm(const GemmParams& p, int64_t tiles_upper_bound, const DeviceInfo& dev,
                     cudaStream_t stream) {
  const size_t smem = gemm_smem_bytes(p.E);
  // per-device set-up, cached (a race between host threads only repeats it)
  static std::atomic<int> configured[kMaxDevices] = {};
  static std::atomic<int> max_pairs[kMaxDevices] = {};
  if (!configured[dev.ordinal].load()) {
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, KH, CG>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)gemm_smem_bytes(kMaxExperts));
    if (err != cudaSuccess) return err;
    configured[dev.ordinal].store(1);
  }
  if (CG == 1) {
    int64_t grid = tiles_upper_bound < dev.num_sms ? tiles_upper_bound : dev.num_sms;
    if (grid < 1) grid = 1;
    return launch_pdl(grouped_gemm_kernel<MODE, KH, CG>, dim3((unsigned)grid), dim3(Traits<MODE, KH, CG>::kThreads),
                      smem, stream, 1, p);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(Traits<MODE, KH, CG>::kThreads);
  cfg.dynamicSmemBytes = gemm_smem_bytes(kMaxExperts);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!max_pairs[dev.ordinal].load()) {
    cfg.gridDim = dim3((unsigned)dev.num_sms);
    int n = 0;
    cudaError_t err = cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<MODE, KH, CG>, &cfg);
    if (err != cudaSuccess) return err;
    max_pairs[dev.ordinal].store(n > 0 ? n : 1);
  }
  const int64_t mp = max_pairs[dev.ordinal].load();
  int64_t pairs = tiles_upper_bound < mp ? tiles_upper_bound : mp;
  if (pairs < 1) pairs = 1;
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  cfg.dynamicSmemBytes = smem;
  cfg.numAttrs = g_pdl.load(std::memory_order_relaxed) ? 2 : 1;   // the occupancy query used the cluster alone
  return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<MODE, KH, CG>, p);
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_cols,
              int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(cols * 2)};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode_tensor_map_2d_bf16(map, base, dims, strides, box, estr);
}

void fill_common(GemmParams& p, const int32_t* offsets, int64_t R, int64_t E, int64_t I,
                 const DeviceInfo& dev) {
  p.offsets = offsets;
  p.gidx = nullptr;
  p.aux = nullptr;
  p.wrow = nullptr;
  p.out = nullptr;
  p.out_gu = nullptr;
  p.out_hw = nullptr;
  p.out_part = nullptr;
  p.status = dev.status;
  p.wait_limit_ns = dev.wait_limit_ns;
  p.stall_producer = dev.test_stall_producer;
  p.rows = (int)R;
  p.E = (int)E;
  p.I = (int)I;
  p.K = 0;
  p.n_out = 0;
  p.m_w = 0;
  p.nt = 0;
  p.mt_w = 0;
  p.ldo = 0;
}

template <int MODE, int KH, int CG>
int64_t mgrouped_tile_bound(int64_t R, int64_t E, int nt) {
  constexpr int bm = Traits<MODE, KH, CG>::kBM;
  return ((R + bm - 1) / bm + E) * nt;
}

// CTA pairs (2-SM MMAs, 256-row tiles with 128-row tails) for the M-grouped
// GEMMs as selected by moe_set_gemm_pairs: mode 1 for all of them, modes 2
// and 3 for the forward gate_up GEMM only; and for the weight-gradient GEMMs
// (256-row tiles: two halves on one CTA, or one per CTA of a pair) in mode 3.
bool use_pair(const DeviceInfo& dev, bool gate_up) {
  return dev.gemm_pairs == 1 || (gate_up && (dev.gemm_pairs == 2 || dev.gemm_pairs == 3));
}
bool use_pair_wgrad(const DeviceInfo& dev) { return dev.gemm_pairs == 3; }

// Single-CTA M-grouped GEMMs with a plain bf16 epilogue take 256-row tiles
// once experts average 256 rows or more, else 128-row tiles: with fewer row
// tiles per expert, tiles of one and two halves mixed in a static
// round-robin leave some SMs with twice the work of others.  Measured on the
// Qwen3-MoE shape (256 rows per expert), the down GEMM: 111.5 us on 256-row
// tiles against 113.9 us on 128-row tiles.
template <int MODE>
cudaError_t run_bf16_mgrouped(const GemmParams& p, int64_t R, int64_t E, const DeviceInfo& dev,
                              cudaStream_t stream) {
  if (R >= 256 * E) return run_gemm<MODE, 2, 1>(p, mgrouped_tile_bound<MODE, 2, 1>(R, E, p.nt), dev, stream);
  return run_gemm<MODE, 1, 1>(p, mgrouped_tile_bound<MODE, 1, 1>(R, E, p.nt), dev, stream);
}


}  // namespace

// K split of the router GEMM: the largest divisor of its 64-wide K blocks up
// to 4.  It sets the order in which each logit's fp32 partial sums add up,
// so it depends on H alone: a token's logits do not depend on how many
// tokens are routed with it (nor the workspace size on the device).
int router_parts(int64_t T, int64_t H, int64_t E) {
  (void)T;
  (void)E;
  const int64_t kb = 3 * H / BK;          // 64-wide K blocks of the stacked split weight
  for (int cand = 4; cand > 1; --cand)
    if (kb % cand == 0) return cand;
  return 1;
}

int launch_router_logits(const uint16_t* x, const uint16_t* w_split, int64_t T, int64_t H, int64_t E,
                         int parts, float* part_out, const DeviceInfo& dev, cudaStream_t stream) {
  if (T == 0) return 0;
  GemmParams p;
  fill_common(p, nullptr, T, parts, H, dev);
  if (!make_map(&p.tmA, x, T, H, 64, BMH) || !make_map(&p.tmB, w_split, 3 * H, E, 64, 64)) return -1;
  p.out_part = part_out;
  p.K = (int)(3 * H / parts);   // K extent of one part
  p.n_out = (int)E;
  p.mt_w = (int)((T + BMH - 1) / BMH);
  p.nt = (int)((E + Traits<ROUTER, 1, 1>::kBN - 1) / Traits<ROUTER, 1, 1>::kBN);
  p.ldo = E;
  return run_gemm<ROUTER, 1, 1>(p, (int64_t)parts * p.mt_w * p.nt, dev, stream) == cudaSuccess ? 0 : 1;
}

int launch_gemm_gate_up(const uint16_t* x, const int32_t* src_row, const int32_t* offsets,
                        const uint16_t* gate_up, int64_t T, int64_t R, int64_t H, int64_t E,
                        int64_t I, uint16_t* h, const float* w_perm, float* gu_pre, uint16_t* h_w,
                        const DeviceInfo& dev, cudaStream_t stream) {
  if (R == 0) return 0;
  GemmParams p;
  fill_common(p, offsets, R, E, I, dev);
  // gathered rows: one-row boxes for tile::gather4; rows in order: 128-row
  // boxes, one per half
  const bool ok_a = src_row ? make_map(&p.tmA, x, T, H, 64, 1) : make_map(&p.tmA, x, R, H, 64, BMH);
  if (!ok_a || !make_map(&p.tmB, gate_up, E * H, 2 * I, 64, 64)) return -1;
  p.gidx = src_row;
  p.out = h;
  p.wrow = w_perm;
  p.out_gu = gu_pre;
  p.out_hw = h_w;
  p.K = (int)H;
  p.n_out = (int)I;
  p.nt = (int)((I + 127) / 128);
  p.ldo = I;
  const cudaError_t err =
      use_pair(dev, true) ? run_gemm<FWD_GATEUP, 1, 2>(p, mgrouped_tile_bound<FWD_GATEUP, 1, 2>(R, E, p.nt), dev, stream)
                     : run_gemm<FWD_GATEUP, 1, 1>(p, mgrouped_tile_bound<FWD_GATEUP, 1, 1>(R, E, p.nt), dev, stream);
  return err == cudaSuccess ? 0 : 1;
}

int launch_gemm_down(const uint16_t* h, const int32_t* offsets, const uint16_t* down, int64_t R,
                     int64_t H, int64_t E, int64_t I, uint16_t* y_perm, const DeviceInfo& dev,
                     cudaStream_t stream) {
  if (R == 0) return 0;
  GemmParams p;
  fill_common(p, offsets, R, E, I, dev);
  if (!make_map(&p.tmA, h, R, I, 64, BMH) || !make_map(&p.tmB, down, E * I, H, 64, 64)) return -1;
  p.out = y_perm;
  p.K = (int)I;
  p.n_out = (int)H;
  p.nt = (int)((H + BN - 1) / BN);
  p.ldo = H;
  const cudaError_t err =
      use_pair(dev, false) ? run_gemm<FWD_DOWN, 1, 2>(p, mgrouped_tile_bound<FWD_DOWN, 1, 2>(R, E, p.nt), dev, stream)
                     : run_bf16_mgrouped<FWD_DOWN>(p, R, E, dev, stream);
  return err == cudaSuccess ? 0 : 1;
}

int down_bwd_parts(int64_t I) { return (int)((I + 63) / 64); }   // one per 64 columns of I

int launch_gemm_down_bwd(const uint16_t* dy_perm, const uint16_t* h_w, const float* gu_pre,
                         const float* w_perm, const int32_t* offsets, const uint16_t* down, int64_t R,
                         int64_t H, int64_t E, int64_t I, uint16_t* dgu, uint16_t* d_down,
                         float* dw_part, const DeviceInfo& dev, cudaStream_t stream) {
  if (R > 0) {  // dgu = SwiGLU'(w * (dy_perm . Wd_e^T), gu_pre)
    GemmParams p;
    fill_common(p, offsets, R, E, I, dev);
    const bool pair = use_pair(dev, false);   // a pair's CTA loads 128 of the tile's 256 B rows
    if (!make_map(&p.tmA, dy_perm, R, H, 64, BMH) || !make_map(&p.tmB, down, E * I, H, 64, pair ? 128 : 256))
      return -1;
    p.aux = gu_pre;
    p.wrow = w_perm;
    p.out = dgu;
    p.out_part = dw_part;
    p.K = (int)H;
    p.n_out = (int)I;
    p.nt = (int)((I + BN - 1) / BN);
    p.ldo = 2 * I;
    const cudaError_t err =
        pair ? run_gemm<DGRAD_DOWN, 1, 2>(p, mgrouped_tile_bound<DGRAD_DOWN, 1, 2>(R, E, p.nt), dev, stream)
             : run_gemm<DGRAD_DOWN, 1, 1>(p, mgrouped_tile_bound<DGRAD_DOWN, 1, 1>(R, E, p.nt), dev, stream);
    if (err != cudaSuccess) return 1;
  }
  {  // d_down_e = (w h)_e^T . dy_perm_e
    GemmParams p;
    fill_common(p, offsets, R, E, I, dev);
    const int64_t rows = R > 0 ? R : 1;
    if (!make_map(&p.tmA, h_w, rows, I, 64, 64) || !make_map(&p.tmB, dy_perm, rows, H, 64, 64))
      return -1;
    p.out = d_down;
    p.m_w = (int)I;
    p.n_out = (int)H;
    p.mt_w = (int)((I + 2 * BMH - 1) / (2 * BMH));
    p.nt = (int)((H + BN - 1) / BN);
    p.ldo = H;
    const cudaError_t err = use_pair_wgrad(dev) ? run_gemm<WGRAD_DOWN, 1, 2>(p, E * p.mt_w * p.nt, dev, stream)
                                                : run_gemm<WGRAD_DOWN, 2, 1>(p, E * p.mt_w * p.nt, dev, stream);
    if (err != cudaSuccess) return 1;
  }
  return 0;
}

int launch_gemm_gate_up_bwd(const uint16_t* dgu, const uint16_t* x, const int32_t* src_row,
                            const int32_t* offsets, const uint16_t* gate_up, int64_t T, int64_t R,
                            int64_t H, int64_t E, int64_t I, uint16_t* dx_perm,
                            uint16_t* d_gate_up, const DeviceInfo& dev, cudaStream_t stream) {
  if (R > 0) {  // dx_perm = dgu . Wgu_e^T
    GemmParams p;
    fill_common(p, offsets, R, E, I, dev);
    const bool pair = use_pair(dev, false);
    if (!make_map(&p.tmA, dgu, R, 2 * I, 64, BMH) ||
        !make_map(&p.tmB, gate_up, E * H, 2 * I, 64, pair ? 128 : 256))
      return -1;
    p.out = dx_perm;
    p.K = (int)(2 * I);
    p.n_out = (int)H;
    p.nt = (int)((H + BN - 1) / BN);
    p.ldo = H;
    const cudaError_t err =
        pair ? run_gemm<DGRAD_GATEUP, 1, 2>(p, mgrouped_tile_bound<DGRAD_GATEUP, 1, 2>(R, E, p.nt), dev, stream)
             : run_bf16_mgrouped<DGRAD_GATEUP>(p, R, E, dev, stream);
    if (err != cudaSuccess) return 1;
  }
  {  // d_gate_up_e = x[rows of e]^T . dgu_e
    GemmParams p;
    fill_common(p, offsets, R, E, I, dev);
    const int64_t rows = R > 0 ? R : 1;
    const bool ok_a = src_row ? make_map(&p.tmA, x, T > 0 ? T : 1, H, 64, 1)
                              : make_map(&p.tmA, x, rows, H, 64, 64);
    if (!ok_a || !make_map(&p.tmB, dgu, rows, 2 * I, 64, 64)) return -1;
    p.gidx = src_row;
    p.out = d_gate_up;
    p.m_w = (int)H;
    p.n_out = (int)(2 * I);
    p.mt_w = (int)((H + 2 * BMH - 1) / (2 * BMH));
    p.nt = (int)((2 * I + BN - 1) / BN);
    p.ldo = 2 * I;
    const cudaError_t err = use_pair_wgrad(dev) ? run_gemm<WGRAD_GATEUP, 1, 2>(p, E * p.mt_w * p.nt, dev, stream)
                                                : run_gemm<WGRAD_GATEUP, 2, 1>(p, E * p.mt_w * p.nt, dev, stream);
    if (err != cudaSuccess) return 1;
  }
  return 0;
}

}  // namespace moe
