// attn_fwd.cuh -- blockwise DiT attention forward for sm_103a.
//
// What it computes ("xDiT: an Inference Engine for DiTs with Massive
// Parallelism", abstract; "SwiftFusion: Scalable Sequence Parallelism ...",
// ideas 1-2): for every (batch, head) and query row i,
//     O_i = sum_j softmax_j(q_i . k_j / sqrt(D)) v_j,  LSE_i = ln sum_j exp(...)
// with the keys split into n contiguous chunks [floor(cS/n), floor((c+1)S/n)).
// Each chunk yields (O_c, LSE_c); they are folded into the running result by
// log-sum-exp weights, so any chunk count reproduces unchunked attention.
//
// Design (one CTA = one (batch*head, pair of 128-row query tiles)):
//   warp 0      TMA producer: Q tiles once, then K and V tiles (128 keys each)
//               through NS-stage shared-memory rings.
//   warp 1      allocates 512 TMEM columns and issues every tcgen05
//               instruction: S_t = Q_t K^T (SS form, fp32 in TMEM) and
//               O_t += P_t V (TS form: P read from TMEM, V from shared memory).
//               The whole warp runs the issue loop with warp-uniform operands
//               and one elected lane executes each MMA and commit; issuing
//               from a single lane inside a divergent branch cost about twice
//               as many cycles per MMA.
//   warps 2-5   softmax for query tile 0, warps 6-9 for query tile 1.  Each
//               thread owns one query row (one TMEM lane): it loads its S row
//               with the reducing TMEM load that also returns the row max
//               (sm_103a), rescales its O row in TMEM when the
//               reference max has to move, writes P = 2^(S*scale - m) as bf16
//               and keeps the row sum.
// TMEM columns: S_t at 128 t.  D = 64: O_t at 256 + 64 t and P_t at
// 384 + 64 t, so S_t of the next key tile is computed as soon as the softmax
// has loaded S_t into registers (QK^T runs while the softmax works) and only
// the PV that reads P_t has to wait for it.  D = 72: room for the P columns
// of one query tile: O_0 at 256, O_1 at 352, P_0 at 448; tile 1 writes P_1
// over the first 64 columns of S_1, so its QK^T of the next key tile follows
// its PV of this one.  D = 128: no room for P on its own; O_t at 256 + 128 t
// and P_t over the first 64 columns of S_t.
// The two softmax groups ping-pong: while one group works on its tile the
// tensor core runs the other tile's MMAs.
//
// Online softmax in base 2: x = S * log2(e) / sqrt(D).  The reference max m
// only moves when a tile's max exceeds it by more than kRescaleThreshold, so
// P <= 2^kRescaleThreshold and O is rescaled rarely; the result is exact up to
// rounding because O and the row sum l always share the same reference.
//
// Chunk merge on chip: every chunk's partial result is accumulated against
// one shared reference max m and left unnormalised.  With
// l_c = sum_{j in c} 2^(x_j - m) the chunk's row sum, the accumulator holds
// A = sum_c A_c, A_c = sum_{j in c} 2^(x_j - m) v_j = l_c O_c, and each
// finished chunk's log2-LSE, LSE_c = m + log2(l_c), is folded into the
// running L = log2(2^L + 2^LSE_c).  The log-sum-exp merge of the normalised
// partials, O = sum_c 2^(LSE_c - L) O_c = 2^(m - L) sum_c A_c, is therefore
// one scale of the accumulator by 2^(m - L) at the end: no pass over O is
// made at a chunk boundary, and the largest weight of a row stays exactly 1
// when it sets the reference.  When m moves, the accumulator and the open
// chunk's l_c are rescaled together; L is absolute and never rescaled.
// Two key walks.  Chunk by chunk (the default): key tiles never straddle
// chunks; a tile that would is cut at the chunk end (columns past it are
// masked to -inf) and the next chunk starts a new tile.  Grid walk (kGrid,
// every chunk at least one tile long): the tiles lie on the global 128-key
// grid and a tile that straddles a chunk end is computed once; its PV is
// shared (same reference, same accumulator) and only its row sum is split at
// the chunk end: the smaller side is summed again with the same instructions,
// the other side is the rest.  With chunks of at least one tile, a tile holds
// at most one chunk end.
//
// Epilogue of the merged result: each thread scales its O row by 2^(m - L)
// and rounds it to bf16.  At D = 72 a warp stages its 32 rows in shared
// memory (over its group's Q tile, whose last QK^T has completed) and writes
// them with one TMA store; the per-thread row stores it replaces touch 32
// rows per instruction, which cost DiT-XL/2 about 4 % of its launch.  At
// D = 64 and 128 the per-thread stores measured as fast or faster, and stay.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace ditk {

constexpr int kBlockM = 128;           // query rows per tile = TMEM lanes
constexpr int kBlockN = 128;           // keys per K/V tile
constexpr int kAttnThreads = 320;      // 10 warps
constexpr int kSwzBytes = kBlockM * 128;  // one 64-column SW128 block of 128 rows
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kLog2e = 1.442695040888963407f;

// Per head-dimension layout.  The head dimension is the MMA K of QK^T and the
// MMA N of PV.  Columns 0..63 live in a 128-byte-swizzled block; the rest in a
// second block: 64 columns (D = 128, 128-byte swizzle) or, for Q and K with
// D = 72, 16 columns (32-byte swizzle; one more K = 16 step of QK^T).  V with
// D = 72 carries a full 128-byte-swizzled block from column 64, so that PV is
// a single N = 80 MMA per 16 keys.  TMA zero-fills every column past 71, so
// padding D to 80 is exact.
template <int D>
struct AttnCfg;
template <>
struct AttnCfg<64> {
  static constexpr int kDpad = 64, kTail = 0, kVTail = 0, kStages = 4;
};
// D = 72 runs two K/V stages: against three, DiT-XL/2 (eight key tiles a
// CTA) gains 2-3 % and PixArt is unchanged; D = 64 loses 2.6 % with three
// stages instead of four.
template <>
struct AttnCfg<72> {
  static constexpr int kDpad = 80, kTail = 16, kVTail = 64, kStages = 2;
};
template <>
struct AttnCfg<128> {
  static constexpr int kDpad = 128, kTail = 64, kVTail = 64, kStages = 2;
};

template <int D>
struct AttnLayout {
  using C = AttnCfg<D>;
  static constexpr int kTileBytes = kSwzBytes + kBlockM * C::kTail * 2;    // a Q or K tile
  static constexpr int kVTileBytes = kSwzBytes + kBlockM * C::kVTail * 2;  // a V tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + C::kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + C::kStages * kVTileBytes;
  static constexpr int kNumBars = 2 + 4 * C::kStages + 11;
  static constexpr int kTmemSlotOff = kBarOff + 8 * kNumBars;
  static constexpr int kBytes = kTmemSlotOff + 16;
  static constexpr int kSmemLaunch = kBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kTileBytes % 1024 == 0 && kVTileBytes % 1024 == 0, "tiles must keep 1024-byte alignment");
  static_assert(kSmemLaunch <= 232448, "shared memory budget");
};

struct AttnParams {
  __nv_bfloat16 *out;  // merged mode: bf16 [BH, S, D]
  float *lse;          // merged mode: fp32 [BH, S] or nullptr
  float *partials;     // partials mode: fp32 [n, BH*S, D]
  float *part_lse;     // partials mode: fp32 [n, BH*S]
  long long rows_total;  // BH * S
  int S;
  int n_chunks;
  int num_pairs;       // ceil(ceil(S / 128) / 2)
  int tiles_total;     // merged mode: number of key tiles over all chunks
  int key_j0, key_j1;  // partials mode with key_j1 > 0: one key range, written to slot 0
  int chunk_q, chunk_r;  // S = chunk_q * n_chunks + chunk_r (merged mode's chunk walk)
  int pair_units;      // merged mode: CTAs below this index take a pair of query tiles; each
                       // later pair is split into two CTAs of one query tile (the last wave)
  float scale_log2;    // log2(e) / sqrt(D)
};

// Walks the key tiles chunk by chunk: every chunk starts a new tile and a
// tile stops at its chunk's end (columns past it are masked).  Chunk c covers
// [floor(c S / n), floor((c + 1) S / n)); the chunk ends are stepped without
// a division: with S = q n + r, chunk c ends q keys after the previous end,
// plus one when the running remainder (c + 1) r mod n wraps past n.  q, r and
// n stay in the kernel parameters; a single key range is one chunk.
struct KvIter {
  int j0, j1;  // current chunk [j0, j1)
  int t0;      // first key of the current tile
  int rem;     // (c + 1) r mod n for the current chunk c
  __device__ __forceinline__ void start(int q, int r) {
    j0 = 0;
    j1 = q;
    t0 = 0;
    rem = r;
  }
  // A single explicit key range [j0_, j1_).
  __device__ __forceinline__ void start_range(int j0_, int j1_) {
    j0 = j0_;
    j1 = j1_;
    t0 = j0_;
    rem = 0;
  }
  __device__ __forceinline__ int valid() const { return min(kBlockN, j1 - t0); }
  __device__ __forceinline__ bool chunk_start() const { return t0 == j0; }
  // Moves the chunk bounds on to the next chunk.
  __device__ __forceinline__ void step_chunk(int q, int r, int n) {
    j0 = j1;
    j1 += q;
    rem += r;
    if (rem >= n) {
      rem -= n;
      ++j1;
    }
  }
  // q, r, n: the partition (S = q n + r); unused once the last chunk is done.
  __device__ __forceinline__ void next(int q, int r, int n) {
    t0 += kBlockN;
    if (t0 >= j1) {
      step_chunk(q, r, n);
      t0 = j0;
    }
  }
};

__device__ __forceinline__ float logaddexp2(float a, float b) {
  const float mx = fmaxf(a, b), mn = fminf(a, b);
  if (mn == -INFINITY) return mx;
  return mx + lg2_approx(1.0f + ex2_approx(mn - mx));
}

// ------------------------------------------------------------ MMA issue
// Shared-memory descriptors as (low, high) words: the high word is fixed per
// operand layout, and stepping along K or to another stage is one add on the
// low word.
constexpr uint32_t kHi128 = desc_hi(1024, kSwizzle128B);
constexpr uint32_t kHi32 = desc_hi(256, kSwizzle32B);

template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tS, uint32_t q_lo, uint32_t k_lo) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBlockM, kBlockN, false);
  constexpr uint32_t kBlk = kSwzBytes >> 4;
  if constexpr (D == 128) {
    // Both 64-column blocks of the head dimension, four K = 16 steps each, in
    // two issue blocks (one elected lane, descriptors stepped in registers):
    // fewer instructions on the issuing warp's sub-partition, which it shares
    // with two softmax warps (+3 % on Flux; at D = 64 and 72 the per-MMA form
    // measured as fast or faster and stays).
    umma_ss4_e(tS, desc64(q_lo, kHi128), desc64(k_lo, kHi128), idesc, 0u);
    umma_ss4_e(tS, desc64(q_lo + kBlk, kHi128), desc64(k_lo + kBlk, kHi128), idesc, 1u);
  } else {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      umma_ss_e(tS, q_lo + 2 * ks, kHi128, k_lo + 2 * ks, kHi128, idesc, ks > 0 ? 1u : 0u);
    if constexpr (D == 72) umma_ss_e(tS, q_lo + kBlk, kHi32, k_lo + kBlk, kHi32, idesc, 1u);
  }
}

// O (+)= P V: P is bf16 in TMEM (8 columns per 16 keys), V is MN-major in
// shared memory (rows = keys, 128 bytes per row per 64-column block).  One
// MMA of N = Dpad per 16 keys; v_lo carries the leading byte offset from one
// 64-column block of V to the next.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint32_t v_lo, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBlockM, AttnCfg<D>::kDpad, true);
  if constexpr (D == 128) {
    umma_ts8_e(tO, tP, desc64(v_lo, kHi128), idesc, accumulate ? 1u : 0u);
  } else {
#pragma unroll
    for (int ks = 0; ks < kBlockN / 16; ++ks) {
      const uint32_t acc = (accumulate || ks > 0) ? 1u : 0u;
      umma_ts_e(tO, tP + ks * 8, v_lo + ks * (2048 >> 4), kHi128, idesc, acc);
    }
  }
}

// Multiplies this thread's O row (Dpad fp32 columns in TMEM) by f.  Not waited.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tO, float f) {
  constexpr int kFull = AttnCfg<D>::kDpad / 32;
#pragma unroll
  for (int cb = 0; cb < kFull; ++cb) {
    uint32_t r[32];
    tmem_ld32_wait(tO + cb * 32, r);
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
    tmem_st32(tO + cb * 32, r);
  }
  if constexpr (AttnCfg<D>::kDpad % 32 == 16) {
    uint32_t r[16];
    tmem_ld16_wait(tO + kFull * 32, r);
#pragma unroll
    for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
    tmem_st16(tO + kFull * 32, r);
  }
}

// Writes `count` fp32 values times `sc` as bf16 (count % 8 == 0) to dst.
__device__ __forceinline__ void store_bf16_row(__nv_bfloat16 *dst, const uint32_t *r, int count,
                                               float sc) {
  for (int j = 0; j < count; j += 8) {
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(r[j + 0]) * sc, __uint_as_float(r[j + 1]) * sc);
    v.y = pack_bf16x2(__uint_as_float(r[j + 2]) * sc, __uint_as_float(r[j + 3]) * sc);
    v.z = pack_bf16x2(__uint_as_float(r[j + 4]) * sc, __uint_as_float(r[j + 5]) * sc);
    v.w = pack_bf16x2(__uint_as_float(r[j + 6]) * sc, __uint_as_float(r[j + 7]) * sc);
    *reinterpret_cast<uint4 *>(dst + j) = v;
  }
}

// The same row, scaled and rounded to bf16, to shared memory at `addr`.
__device__ __forceinline__ void stage_bf16_row(uint32_t addr, const uint32_t *r, int count, float sc) {
  for (int j = 0; j < count; j += 8) {
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(r[j + 0]) * sc, __uint_as_float(r[j + 1]) * sc);
    v.y = pack_bf16x2(__uint_as_float(r[j + 2]) * sc, __uint_as_float(r[j + 3]) * sc);
    v.z = pack_bf16x2(__uint_as_float(r[j + 4]) * sc, __uint_as_float(r[j + 5]) * sc);
    v.w = pack_bf16x2(__uint_as_float(r[j + 6]) * sc, __uint_as_float(r[j + 7]) * sc);
    st_shared_v4(addr + j * 2, v);
  }
}

__device__ __forceinline__ void store_f32_row(float *dst, const uint32_t *r, int count, float sc) {
  for (int j = 0; j < count; j += 4) {
    float4 v = make_float4(__uint_as_float(r[j + 0]) * sc, __uint_as_float(r[j + 1]) * sc,
                           __uint_as_float(r[j + 2]) * sc, __uint_as_float(r[j + 3]) * sc);
    *reinterpret_cast<float4 *>(dst + j) = v;
  }
}

// ------------------------------------------------------------------ kernel
// kPartials = false: all chunks, merged on chip, bf16 O + fp32 LSE.
// kPartials = true : one chunk per CTA, fp32 O_c + LSE_c, no merge.
// kPdl: launched with programmatic stream serialization (see ptx.cuh); the
//   host takes it for grids of a few waves, where the launch gap between
//   kernels is a visible share of the time.  Long grids use the plain launch
//   and a kernel without the two grid-dependency instructions, whose position
//   in the code measurably cost the D = 64 loop about 2 %.
// kGrid (merged mode only): the grid walk described at the top.  A separate
//   instantiation, because its straddle code slows the loop by a few per cent
//   even where it never runs.
template <int D, bool kPartials, bool kPdl, bool kGrid = false>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_q_tail,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_k_tail,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_v_tail,
                    const __grid_constant__ CUtensorMap tm_o, const AttnParams p) {
  using C = AttnCfg<D>;
  using L = AttnLayout<D>;
  constexpr int NS = C::kStages;
  constexpr uint32_t kTileBytes = L::kTileBytes;
  constexpr uint32_t kVTileBytes = L::kVTileBytes;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work unit and its key walk.
  int bh, pair, chunk_first, tiles;
  KvIter kv0;
  int q_tile_in_pair = 0;
  bool single = false;
  if constexpr (kPartials) {
    const int per_bh_chunk = p.num_pairs;
    const int u = blockIdx.x;
    pair = u % per_bh_chunk;
    const int bc = u / per_bh_chunk;
    chunk_first = bc % p.n_chunks;
    bh = bc / p.n_chunks;
    const long long j0 = p.key_j1 > 0 ? p.key_j0 : (static_cast<long long>(chunk_first) * p.S) / p.n_chunks;
    const long long j1 = p.key_j1 > 0 ? p.key_j1 : (static_cast<long long>(chunk_first + 1) * p.S) / p.n_chunks;
    tiles = static_cast<int>((j1 - j0 + kBlockN - 1) / kBlockN);
    kv0.start_range(static_cast<int>(j0), static_cast<int>(j1));
  } else {
    int g = blockIdx.x;
    if (g >= p.pair_units) {
      const int u = g - p.pair_units;
      g = p.pair_units + (u >> 1);
      q_tile_in_pair = u & 1;
      single = true;
    }
    pair = g % p.num_pairs;
    bh = g / p.num_pairs;
    chunk_first = 0;
    tiles = p.tiles_total;
    kv0.start(p.chunk_q, p.chunk_r);
  }
  const int q_row0 = (pair * 2 + q_tile_in_pair) * kBlockM;
  const bool has1 = !single && q_row0 + kBlockM < p.S;

  // Shared-memory addresses.
  const uint32_t sQ0 = base + L::kQOff;
  const uint32_t sK0 = base + L::kKOff;
  const uint32_t sV0 = base + L::kVOff;
  const uint32_t bars = base + L::kBarOff;
  auto q_full = [&](int t) { return bars + 8u * t; };
  auto k_full = [&](int s) { return bars + 8u * (2 + s); };
  auto k_empty = [&](int s) { return bars + 8u * (2 + NS + s); };
  auto v_full = [&](int s) { return bars + 8u * (2 + 2 * NS + s); };
  auto v_empty = [&](int s) { return bars + 8u * (2 + 3 * NS + s); };
  auto s_full = [&](int t) { return bars + 8u * (2 + 4 * NS + t); };
  auto p_full = [&](int t) { return bars + 8u * (4 + 4 * NS + t); };
  auto o_full = [&](int t) { return bars + 8u * (6 + 4 * NS + t); };
  const uint32_t mma_done = bars + 8u * (8 + 4 * NS);
  auto s_free = [&](int t) { return bars + 8u * (9 + 4 * NS + t); };
  auto o_upd = [&](int t) { return bars + 8u * (11 + 4 * NS + t); };
  // s_free(t): the softmax group has loaded S_t (D = 64 only); o_upd(t): the
  // PV of tile t has completed, so P_t and O_t are free (D = 64 only).
  constexpr bool kSplitP = (D == 64);               // both query tiles
  constexpr bool kSplitP0 = (D == 64 || D == 72);   // query tile 0
  // TMEM columns of O_1, P_0, P_1 (O_0 at 256, S_t at 128 t).  D = 72 has room
  // for P columns of one query tile only: O_0 [256, 336), O_1 [352, 432),
  // P_0 [448, 512); P_1 is written over the first 64 columns of S_1.
  constexpr uint32_t kO1 = D == 64 ? 320u : (D == 72 ? 352u : 384u);
  constexpr uint32_t kP0 = D == 64 ? 384u : 448u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kTmemSlotOff);

  if (threadIdx.x == 0) {
    mbar_init(q_full(0), 1);
    mbar_init(q_full(1), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), kBlockM);
      mbar_init(o_full(t), 1);
    }
    mbar_init(mma_done, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_free(t), kBlockM);
      mbar_init(o_upd(t), 1);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if constexpr (C::kTail > 0) {
      tma_prefetch_desc(&tm_q_tail);
      tma_prefetch_desc(&tm_k_tail);
      tma_prefetch_desc(&tm_v_tail);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(tmem_slot);
  if constexpr (kPdl) {
    // The next kernel in the stream may launch now: its CTAs take the SMs
    // this grid leaves idle or frees, run their prologue and wait here.
    // Every global read and write of this grid comes after the wait for the
    // previous kernel to have completed.
    griddep_launch_dependents();
    griddep_wait();
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      for (int t = 0; t < 2; ++t) {
        if (t == 1 && !has1) break;
        const uint32_t dst = sQ0 + t * kTileBytes;
        mbar_arrive_expect_tx(q_full(t), kTileBytes);
        tma_load_3d(dst, &tm_q, q_full(t), 0, q_row0 + t * kBlockM, bh, pol_q);
        if constexpr (C::kTail > 0)
          tma_load_3d(dst + kSwzBytes, &tm_q_tail, q_full(t), 64, q_row0 + t * kBlockM, bh, pol_q);
      }
      KvIter kv = kv0;
      int k_last[NS], v_last[NS];  // last use issued on each stage, -1 if none
#pragma unroll
      for (int s = 0; s < NS; ++s) k_last[s] = v_last[s] = -1;
      for (int it = 0; it < tiles; ++it) {
        const int s = it % NS;
        const int u = it / NS;
        if (u > 0 && !mbar_wait(k_empty(s), (u - 1) & 1)) break;
        const uint32_t kd = sK0 + s * kTileBytes;
        mbar_arrive_expect_tx(k_full(s), kTileBytes);
        tma_load_3d(kd, &tm_k, k_full(s), 0, kv.t0, bh, pol_kv);
        if constexpr (C::kTail > 0) tma_load_3d(kd + kSwzBytes, &tm_k_tail, k_full(s), 64, kv.t0, bh, pol_kv);
        k_last[s] = u;
        if (u > 0 && !mbar_wait(v_empty(s), (u - 1) & 1)) break;
        const uint32_t vd = sV0 + s * kVTileBytes;
        mbar_arrive_expect_tx(v_full(s), kVTileBytes);
        tma_load_3d(vd, &tm_v, v_full(s), 0, kv.t0, bh, pol_kv);
        if constexpr (C::kVTail > 0) tma_load_3d(vd + kSwzBytes, &tm_v_tail, v_full(s), 64, kv.t0, bh, pol_kv);
        v_last[s] = u;
        if constexpr (kGrid) kv.t0 += kBlockN;
        else kv.next(p.chunk_q, p.chunk_r, p.n_chunks);
      }
      // Drain: every load issued must land before the CTA may exit.  Waiting on
      // the parity of a stage's last use returns at once if it already landed.
      // These waits ignore the device status word (see ptx.cuh).
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        if (k_last[s] >= 0) mbar_wait_drain(k_full(s), k_last[s] & 1);
        if (v_last[s] >= 0) mbar_wait_drain(v_full(s), v_last[s] & 1);
      }
      if (has1) mbar_wait_drain(q_full(1), 0);
      mbar_wait_drain(q_full(0), 0);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issue
    // The whole warp runs the loop; one elected lane issues each instruction.
    {
      const uint32_t tS0 = tmem_base, tS1 = tmem_base + 128;
      const uint32_t tO0 = tmem_base + 256, tO1 = tmem_base + kO1;
      const uint32_t tP0 = kSplitP0 ? tmem_base + kP0 : tS0, tP1 = kSplitP ? tmem_base + 448 : tS1;
      const uint32_t q_lo0 = desc_lo(sQ0, 16), k_lo0 = desc_lo(sK0, 16), v_lo0 = desc_lo(sV0, kSwzBytes);
      bool ok = mbar_wait_warp(q_full(0), 0) && (!has1 || mbar_wait_warp(q_full(1), 0));
      tc_fence_after();
      for (int it = 0; ok && it < tiles; ++it) {
        const int s = it % NS, u = it / NS;
        if (!(ok = mbar_wait_warp(k_full(s), u & 1))) break;
        tc_fence_after();
        const uint32_t ks = k_lo0 + s * (kTileBytes >> 4);
        const int ps = (it + NS - 1) % NS;
        const uint32_t vs = v_lo0 + ps * (kVTileBytes >> 4);
        if constexpr (kSplitP) {
          // Per query tile: S_t of this key tile once the softmax has loaded
          // the previous S_t, then the PV of the previous key tile once its
          // P_t is written.
          if (it > 0 && !(ok = mbar_wait_warp(s_free(0), (it - 1) & 1))) break;
          tc_fence_after();
          issue_qk<D>(tS0, q_lo0, ks);
          umma_commit_e(s_full(0));
          if (it > 0) {
            if (!(ok = mbar_wait_warp(p_full(0), (it - 1) & 1))) break;
            if (!(ok = mbar_wait_warp(v_full(ps), ((it - 1) / NS) & 1))) break;
            tc_fence_after();
            issue_pv<D>(tO0, tP0, vs, it > 1);
            umma_commit_e(o_upd(0));
          }
          if (has1) {
            if (it > 0 && !(ok = mbar_wait_warp(s_free(1), (it - 1) & 1))) break;
            tc_fence_after();
            issue_qk<D>(tS1, q_lo0 + (kTileBytes >> 4), ks);
            umma_commit_e(s_full(1));
            if (it > 0) {
              if (!(ok = mbar_wait_warp(p_full(1), (it - 1) & 1))) break;
              tc_fence_after();
              issue_pv<D>(tO1, tP1, vs, it > 1);
              umma_commit_e(o_upd(1));
            }
          }
          umma_commit_e(k_empty(s));
          if (it > 0) umma_commit_e(v_empty(ps));
        } else if constexpr (kSplitP0) {
          // Query tile 0 as above; tile 1 writes P over S, so its QK^T of
          // this key tile follows the PV of the previous one.
          if (it > 0 && !(ok = mbar_wait_warp(s_free(0), (it - 1) & 1))) break;
          tc_fence_after();
          issue_qk<D>(tS0, q_lo0, ks);
          umma_commit_e(s_full(0));
          if (it > 0) {
            if (!(ok = mbar_wait_warp(p_full(0), (it - 1) & 1))) break;
            if (!(ok = mbar_wait_warp(v_full(ps), ((it - 1) / NS) & 1))) break;
            tc_fence_after();
            issue_pv<D>(tO0, tP0, vs, it > 1);
            umma_commit_e(o_upd(0));
          }
          if (has1) {
            if (it > 0) {
              if (!(ok = mbar_wait_warp(p_full(1), (it - 1) & 1))) break;
              tc_fence_after();
              issue_pv<D>(tO1, tP1, vs, it > 1);
            }
            issue_qk<D>(tS1, q_lo0 + (kTileBytes >> 4), ks);
            umma_commit_e(s_full(1));
          }
          if (it > 0) umma_commit_e(v_empty(ps));
          umma_commit_e(k_empty(s));
        } else {
          if (it > 0) {
            if (!(ok = mbar_wait_warp(p_full(0), (it - 1) & 1))) break;
            if (!(ok = mbar_wait_warp(v_full(ps), ((it - 1) / NS) & 1))) break;
            tc_fence_after();
            issue_pv<D>(tO0, tP0, vs, it > 1);
          }
          issue_qk<D>(tS0, q_lo0, ks);
          umma_commit_e(s_full(0));
          if (has1) {
            if (it > 0) {
              if (!(ok = mbar_wait_warp(p_full(1), (it - 1) & 1))) break;
              tc_fence_after();
              issue_pv<D>(tO1, tP1, vs, it > 1);
            }
            issue_qk<D>(tS1, q_lo0 + (kTileBytes >> 4), ks);
            umma_commit_e(s_full(1));
          }
          if (it > 0) umma_commit_e(v_empty(ps));
          umma_commit_e(k_empty(s));
        }
      }
      if (ok) {
        const int ls = (tiles - 1) % NS;
        const uint32_t vs = v_lo0 + ls * (kVTileBytes >> 4);
        ok = mbar_wait_warp(p_full(0), (tiles - 1) & 1) && mbar_wait_warp(v_full(ls), ((tiles - 1) / NS) & 1);
        if (ok) {
          tc_fence_after();
          issue_pv<D>(tO0, tP0, vs, tiles > 1);
          umma_commit_e(o_full(0));
          if (has1 && mbar_wait_warp(p_full(1), (tiles - 1) & 1)) {
            tc_fence_after();
            issue_pv<D>(tO1, tP1, vs, tiles > 1);
            umma_commit_e(o_full(1));
          }
        }
      }
      // Every MMA this warp issued completes before TMEM is freed.
      umma_commit_e(mma_done);
      mbar_wait_drain_warp(mma_done, 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax
    const int t = (warp - 2) >> 2;   // query tile handled by this warpgroup
    const int quarter = warp & 3;    // TMEM lane quarter this warp may access
    const int row_in_tile = quarter * 32 + lane;
    if (t == 0 || has1) {
      const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
      const uint32_t tS = tmem_base + t * 128 + lane_off;
      const uint32_t tO = tmem_base + 256 + t * (kO1 - 256) + lane_off;
      // This group's P columns: its own (split) or over its S columns.
      const bool split = kSplitP || (kSplitP0 && t == 0);
      const uint32_t tP = split ? tmem_base + kP0 + t * 64 + lane_off : tS;
      const float scale_log2 = p.scale_log2;
      float m = -INFINITY;     // reference max, base-2 scaled units
      float l = 0.0f;          // row sum of the current chunk
      float l_run = -INFINITY; // merged log2-LSE of finished chunks
      KvIter kv = kv0;
      bool ok = true;
      for (int it = 0; it < tiles; ++it) {
        if (!(ok = mbar_wait_warp(s_full(t), it & 1))) break;
        tc_fence_after();
        uint32_t sr[128];
        float hw_max;  // max of the 128 loaded columns, from the reducing load
        tmem_ld128_max_wait(tS, sr, hw_max);
        if (split) {
          // S_t is in registers: the next QK^T may overwrite it.
          tc_fence_before();
          mbar_arrive(s_free(t));
        }
        const int valid = kGrid ? min(kBlockN, p.S - kv.t0) : kv.valid();
        float row_max = hw_max;
        if (valid < kBlockN) {
          // A tile cut at a chunk end or at S: the columns past `valid` are
          // masked to -inf and the max is taken again over the rest (eight
          // independent chains of 3-input max).
#pragma unroll
          for (int j = 0; j < kBlockN; ++j)
            if (j >= valid) sr[j] = __float_as_uint(-INFINITY);
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(sr[i]);
#pragma unroll
          for (int j = 8; j < kBlockN; j += 16) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              mx[i] = max3(mx[i], __uint_as_float(sr[j + i]), __uint_as_float(sr[j + 8 + i]));
          }
          row_max = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        }
        const float tmax = row_max * scale_log2;
        float o_scale = 1.0f;
        if (kGrid ? (kv.j1 == kv.t0 && it > 0) : (kv.chunk_start() && it > 0)) {
          // The previous chunk is complete: fold its LSE into the running one.
          // Its partial output is already in the accumulator with the shared
          // reference m, so the O half of the merge is applied at the end.
          l_run = logaddexp2(l_run, m + lg2_approx(fmaxf(l, 0.0f)));
          l = 0.0f;
          if constexpr (kGrid) kv.step_chunk(p.chunk_q, p.chunk_r, p.n_chunks);
        }
        // Grid walk: the open chunk may end strictly inside this tile (at
        // column b_rel); then the tile's row sum is split there.
        const int b_rel = kv.j1 - kv.t0;
        const bool straddle = kGrid && b_rel < valid;
        if (tmax > m + kRescaleThreshold) {
          const float f = ex2_approx(m - tmax);
          o_scale *= f;
          l *= f;
          m = tmax;
        }
        const float neg_m = -m;
        if (split) {
          // P_t and O_t are free once the previous key tile's PV has completed.
          if (it > 0) {
            if (!(ok = mbar_wait_warp(o_upd(t), (it - 1) & 1))) break;
            tc_fence_after();
          }
        }
        // Straddling tile: the sum of P over the smaller side of the chunk end
        // (at most 64 keys), with the same instructions as the loop below, so
        // the same values; the other side is the tile's sum minus it.  8-key
        // groups outside that side are skipped with a warp-uniform branch.
        float part = 0.0f;
        bool left_small = true;
        if constexpr (kGrid) {
          if (straddle) {
            left_small = b_rel <= kBlockN / 2;
            const int lo = left_small ? 0 : b_rel, hi = left_small ? b_rel : valid;
#pragma unroll
            for (int g = 0; g < kBlockN / 8; ++g) {
              if (8 * g + 8 > lo && 8 * g < hi) {
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                  const int j = 8 * g + i;
                  float x0, x1;
                  fma2(x0, x1, __uint_as_float(sr[j]), __uint_as_float(sr[j + 1]), scale_log2, scale_log2, neg_m,
                       neg_m);
                  const float a = ex2_approx(x0);
                  const float b = ex2_approx(x1);
                  part += (j >= lo && j < hi) ? a : 0.0f;
                  part += (j + 1 >= lo && j + 1 < hi) ? b : 0.0f;
                }
              }
            }
          }
        }
        // P = 2^(S * scale - m): the affine part on packed pairs, 2^x on the
        // MUFU, row sum in four packed accumulators, P packed to bf16 pairs.
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int qtr = 0; qtr < 4; ++qtr) {
          uint32_t pr[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float x0, x1;
            fma2(x0, x1, __uint_as_float(sr[qtr * 32 + 2 * j]), __uint_as_float(sr[qtr * 32 + 2 * j + 1]),
                 scale_log2, scale_log2, neg_m, neg_m);
            const float a = ex2_approx(x0);
            const float b = ex2_approx(x1);
            add2(acc[2 * (j & 3)], acc[2 * (j & 3) + 1], a, b);
            pr[j] = pack_bf16x2(a, b);
          }
          tmem_st16(tP + qtr * 16, pr);
        }
        add2(acc[0], acc[1], acc[2], acc[3]);
        add2(acc[4], acc[5], acc[6], acc[7]);
        add2(acc[0], acc[1], acc[4], acc[5]);
        const float l_tile = acc[0] + acc[1];
        if (straddle) {
          // The open chunk ends inside this tile: its LSE takes the keys left
          // of the end, the next chunk starts with the rest.
          const float l_left = left_small ? part : fmaxf(l_tile - part, 0.0f);
          const float l_right = left_small ? fmaxf(l_tile - part, 0.0f) : part;
          l_run = logaddexp2(l_run, m + lg2_approx(fmaxf(l + l_left, 0.0f)));
          l = l_right;
          kv.step_chunk(p.chunk_q, p.chunk_r, p.n_chunks);
        } else {
          l += l_tile;
        }
        // O may be rescaled after P is written: the PV MMA that reads both waits
        // for this warpgroup's arrival below.  Doing it here, once the S values
        // are dead, keeps the row in registers without spilling.
        if (it > 0 && __any_sync(0xffffffffu, o_scale != 1.0f)) rescale_o<D>(tO, o_scale);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full(t));
        if constexpr (kGrid) kv.t0 += kBlockN;
        else kv.next(p.chunk_q, p.chunk_r, p.n_chunks);
      }
      if (ok) ok = mbar_wait_warp(o_full(t), 0);
      if (ok) {
        tc_fence_after();
        const float lse_c = m + lg2_approx(fmaxf(l, 0.0f));
        const float l_new = logaddexp2(l_run, lse_c);
        const float sc = ex2_approx(m - l_new);
        const int row = q_row0 + t * kBlockM + row_in_tile;
        const bool in_range = row < p.S;
        const long long grow = static_cast<long long>(bh) * p.S + row;
        constexpr int kFull = C::kDpad / 32;
        if constexpr (!kPartials && D == 72) {
          // The warp's 32 rows go to shared memory, over this group's Q tile
          // (its last QK^T completed before o_full), then out in one TMA
          // store; rows past S fall outside the tensor map and are dropped,
          // and a box that starts past S is not issued.  The warp waits until
          // the store has read shared memory before the CTA may free it.
          constexpr uint32_t kRowBytes = D * 2;
          const uint32_t stage = sQ0 + t * kTileBytes + quarter * 32 * kRowBytes;
          const uint32_t mine = stage + lane * kRowBytes;
#pragma unroll
          for (int cb = 0; cb < kFull; ++cb) {
            uint32_t r[32];
            tmem_ld32_wait(tO + cb * 32, r);
            stage_bf16_row(mine + cb * 64, r, 32, sc);
          }
          if constexpr (C::kDpad % 32 == 16) {
            uint32_t r[16];
            tmem_ld16_wait(tO + kFull * 32, r);
            stage_bf16_row(mine + kFull * 64, r, D - kFull * 32, sc);
          }
          fence_proxy_async_smem();
          __syncwarp();
          const int row0 = q_row0 + t * kBlockM + quarter * 32;
          if (lane == 0 && row0 < p.S) {
            tma_store_3d(&tm_o, stage, 0, row0, bh);
            bulk_commit_group();
            bulk_wait_read_all();
          }
          __syncwarp();
          if (in_range && p.lse != nullptr) p.lse[grow] = l_new * kLn2;
        } else if constexpr (!kPartials) {
          __nv_bfloat16 *dst = p.out + grow * D;
#pragma unroll
          for (int cb = 0; cb < kFull; ++cb) {
            uint32_t r[32];
            tmem_ld32_wait(tO + cb * 32, r);
            if (in_range) store_bf16_row(dst + cb * 32, r, 32, sc);
          }
          if constexpr (C::kDpad % 32 == 16) {
            uint32_t r[16];
            tmem_ld16_wait(tO + kFull * 32, r);
            if (in_range) store_bf16_row(dst + kFull * 32, r, D - kFull * 32, sc);
          }
          if (in_range && p.lse != nullptr) p.lse[grow] = l_new * kLn2;
        } else {
          float *dst = p.partials + (static_cast<long long>(chunk_first) * p.rows_total + grow) * D;
#pragma unroll
          for (int cb = 0; cb < kFull; ++cb) {
            uint32_t r[32];
            tmem_ld32_wait(tO + cb * 32, r);
            if (in_range) store_f32_row(dst + cb * 32, r, 32, sc);
          }
          if constexpr (C::kDpad % 32 == 16) {
            uint32_t r[16];
            tmem_ld16_wait(tO + kFull * 32, r);
            if (in_range) store_f32_row(dst + kFull * 32, r, D - kFull * 32, sc);
          }
          if (in_range) p.part_lse[static_cast<long long>(chunk_first) * p.rows_total + grow] = l_new * kLn2;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace ditk
