// Scaled FP8 (and BF16) GEMMs on the 5th-generation tensor cores (sm_103a): dense, and the MoE
// grouped GEMM with rows or contraction jagged by expert.
//
//   D[m, n] = sA[m] * sB[n] * sum_k A[m, k] * B[n, k]       (dequant contract: "FP8 Training:
//   Quantization, Autograd, Torchao", section 2; operand layouts: section 4)
//   grouped: per-row sA, per-expert-column sB, rows routed by cumulative offsets ("FP8 training
//   on AMD GPUs with TorchTitan and TorchAO", "Scaling FP8 to MoE Architectures", Figure 3).
//
// Design (persistent; 320 threads per CTA; CG = 1 or 2 CTAs per MMA):
//   CG = 1: one CTA per SM computes 128 x 256 tiles;
//   CG = 2: a cluster of two CTAs (a CTA pair on two SMs) computes 256 x 256 tiles with
//           tcgen05.mma.cta_group::2: each CTA stages its own 128 rows of A and 128 of the 256
//           rows of B, the even CTA issues the MMAs for both, and each CTA's tensor memory
//           holds the accumulator of its own 128 rows. Per CTA a stage is 32 KB instead of
//           48 KB, so the ring is 6 stages deep and B is read from L2 once per pair.
//   warp 0      TMA producer (128-byte swizzle; K blocks of 128 bytes) into the stage ring,
//               guarded by full/empty mbarriers (the pair's full barrier lives in the even CTA
//               and counts both CTAs' bytes);
//   warp 1      allocates 512 TMEM columns; lane 0 of the issuing CTA issues the MMAs (M=128
//               or 256, N=256; K=32 for FP8, K=16 for BF16) into one of two fp32
//               accumulators and commits each stage back to the producers and each finished
//               tile to the epilogues (multicast to both CTAs of a pair);
//   warps 2..9  epilogue: each warp owns 32 TMEM lanes (tile rows) and one half (128 columns)
//               of its CTA's tile; the tile's column scales are staged once in shared memory;
//               tcgen05.ld 32 columns at a time, sA[m] * sB[n] applied once, one rounding to
//               bf16/fp32, masked stores. The second accumulator lets the next tile's MMAs
//               overlap this epilogue.
// Grouped with rows jagged by expert (FP8, pairs): an expert's last tile, when it has fewer than
// 256 rows, is computed transposed: its 256 weight rows are the MMA's M and its rows, rounded up
// to 16, the MMA's N, loaded with a row box of 32, 64 or 128 per CTA. These GEMMs are bound by
// operand traffic from L2, so a short tail costs the bytes and MMAs of its own rows.
// Every wait is bounded; on a timeout the kernel raises FP8_DEV_TIMEOUT, drains in-flight TMA
// and MMA work, frees its tensor memory and returns.
#include <string.h>

#include "common.cuh"
#include "internal.h"

namespace fp8lin {

namespace {

constexpr int BM = 128, BN = 256, BKB = 128;  // rows per CTA, tile columns (FP8 / BF16), K bytes per stage
constexpr int kTmemCols = 512;
constexpr int kMaxExperts = 2048;
constexpr int64_t kGroupBytes = 32ll << 20;  // rasterization: the A panels of a group of M-blocks, in L2
constexpr int kStageOut = 4096;  // per epilogue warp: output staging for TMA stores (pairs)
// Waits for work already in flight (TMA loads, MMAs) before tensor memory is freed or the CTA
// leaves use this fixed bound, not the adjustable one, so a short limit never frees resources
// under running hardware.
constexpr uint64_t kDrainNs = 2000000000ull;

// kDenseAmax: the dense schedule whose epilogue also folds max |out| into the side outputs;
// kDenseQuant: the dense schedule whose epilogue writes the next quantization of the (bf16) result:
// FP8 codes and 1 x 128 or MX scales along the rows
enum { kDense = 0, kJagM = 1, kJagK = 2, kDenseAmax = 3, kDenseQuant = 4 };
constexpr bool is_dense(int sched) { return sched == kDense || sched == kDenseAmax || sched == kDenseQuant; }
// kBLK: FP8 operands with blockwise scales (A: 1 x 128 tiles, B: 128 x 128 tiles); the MMAs of
// each 128-deep K block go to a fresh tensor-memory partial, which the epilogue warps scale by
// sA[m, kb] * sB[n / 128, kb] and add into register accumulators ("promotion")
enum { kFP8 = 0, kBF16 = 1, kMX = 2, kBLK = 3 };

// MX (block-scaled) tiles are 256 columns wide like the FP8 ones (an MMA's cost is set per
// instruction, so narrower tiles run the tensor cores below their rate), but they keep ONE
// accumulator: its 256 tensor-memory columns plus one 16-column scale-factor slot per ring stage
// fit in the 512 columns, two accumulators would not. Sixteen epilogue warps (four per lane
// quarter, 64 columns each) move the accumulator into registers right after the tile's MMAs and
// release it at once, so the next tile's MMAs wait only for those loads, not for the stores.
template <int KIND, int CG, int SCHED = 0>
struct Cfg {
  // kBLK: single-CTA 128 x 256 tiles and two K-block partials (the MMAs run one K block ahead
  // of the promotion). 128-column tiles with four partials were slower: the MMA's cost is per
  // instruction, so halving N halves the tensor-core rate.
  static constexpr int TBN = BN;                          // tile columns
  static constexpr int NBUF = KIND == kMX ? 1 : 2;        // accumulators / K-block partials
  static constexpr int EPI_WARPS = (KIND == kMX || KIND == kBLK) ? 16 : 8;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  // MX: the warp that copies scales to tensor memory; kBLK: the warp that stages each K block's
  // tile scales in shared memory ahead of the promotion
  static constexpr int SF_WARP = 2 + EPI_WARPS;
  static constexpr int THREADS = 64 + EPI_THREADS + ((KIND == kMX || KIND == kBLK) ? 32 : 0);
  static constexpr int WCOLS = TBN * 4 / EPI_WARPS;      // columns per epilogue warp: 128 or 64
  static constexpr int A_BYTES = BM * BKB;               // this CTA's 128 rows of A
  static constexpr int B_ROWS = TBN / CG;                // this CTA's rows of B
  static constexpr int B_BYTES = B_ROWS * BKB;
  static constexpr int SF_BYTES = KIND == kMX ? 3 * 512 : 0;  // one A scale block, two B scale blocks
  static constexpr int TX_BYTES = A_BYTES + B_BYTES + SF_BYTES;  // bytes the loads of a stage deliver
  static constexpr int STAGE_BYTES = (TX_BYTES + 1023) / 1024 * 1024;
  // MX with the contraction jagged: short K loops make the epilogue's stores the critical path,
  // so those tiles store through shared memory with TMA (64 KB of staging for 16 warps), which
  // leaves room for 4 stages; the other MX schedules store from registers and keep 5
  static constexpr bool MX_TMA_OUT = KIND == kMX && CG == 2 && SCHED == 2;
  static constexpr int STAGES = (CG == 2 && !MX_TMA_OUT) ? 5 : 4;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int OUT_BYTES = (CG == 2 && ((KIND != kMX && KIND != kBLK) || MX_TMA_OUT)) ? EPI_WARPS * kStageOut : 0;
  static constexpr int TILE_M = BM * CG;
  static constexpr int SF_COL0 = NBUF * TBN;             // first scale-factor slot (16 columns each)
};
static_assert(Cfg<kMX, 2>::SF_COL0 + 16 * Cfg<kMX, 2>::STAGES <= kTmemCols, "MX tensor-memory budget");
static_assert(Cfg<kMX, 2, 2>::STAGES <= Cfg<kMX, 2>::STAGES, "MX jagged-K ring");

struct GemmParams {
  int64_t M, N, K;     // tile space: rows of D, columns of D, contraction length (elements)
  int64_t num_m, num_n;
  int64_t nkb;         // K blocks per tile (dense, jagged M)
  int64_t group_m;     // dense: tiles walk group_m M-blocks per N-block (group_n == 0), or
  int64_t group_n;     //        group_n N-blocks per M-block
  const float* sA;
  const float* sB;
  int sa_scalar, sb_scalar;
  void* out;
  int out_f32;
  int vec_ok;          // 16-byte aligned output rows
  int64_t ldo;         // output row stride (elements)
  const int32_t* ends;
  int E;
  int64_t total_rows;  // jagged M: last valid offset
  int tma_out;         // CTA pairs with 16-byte aligned output rows: TMA bulk-tensor stores
  int test_stall;      // wait first on a barrier nothing signals (failure-detection tests)
  uint32_t* row_amax;  // side outputs (bf16 out): max |out| per row / column as fp32 words
  uint32_t* col_amax;
  int amax_whole;      // col_amax is a single word: the maximum over the whole output
  uint32_t idesc;
  int32_t* status;
  uint64_t wait_ns;
  // kDenseQuant: the result's quantization (codes [M, N] row-major in q_fmt; scales: fp32 [M, N / 128]
  // for 1 x 128 blocks, or E8M0 bytes in the MX scale layout for rows M, contraction N)
  uint8_t* q_out;
  void* q_scales;
  int q_mx;
  int q_fmt;
  ScaleTab q_tab;
  // FP8 jagged M on CTA pairs: an expert's last tile, when it holds fewer than 256 rows, is
  // computed transposed (weight rows on the MMA's M side, the tile's rows as its N)
  int tail_t;
  uint32_t idesc_t;    // the transposed tile's instruction descriptor, N field zero
};

struct Tile {
  int64_t m0, n0;   // first row / column of the (pair's) tile of D
  int64_t pm0;      // m0 in the segment-padded row space of the MX A scales (jagged M), else m0
  int64_t row_end;  // rows >= row_end are masked (segment end, or M)
  int64_t k0;       // first contraction coordinate
  int64_t nkb;      // K blocks
  int e;            // expert (jagged)
  int tt;           // jagged M, transposed tail tile: its rows (1..255); 0 for an ordinary tile
};

constexpr int kMaxStages = 5;  // ring stages the barrier arrays below hold
struct Shared {
  float sb[2][BN];  // per-tile column scales, alternating between consecutive tiles
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[4];   // accumulators / K-block partials ready (NBUF of them in use)
  uint64_t tempty[4];
  uint64_t drain;
  uint64_t never;   // signalled by no one: the failure-detection test hook waits on it
  uint64_t sff[kMaxStages];  // MX: a stage's scales are in tensor memory
  uint64_t sf_drain;
  uint32_t tmem_base;
  int abort;
};
constexpr int kSharedBytes = 2304;
// kBLK: a ring of K-block tile scales in shared memory, filled by the scale warp ahead of the
// promotion: per slot this CTA's 128 row scales and the tile's two 128-column block scales
constexpr int kScGroup = 8;   // K blocks whose scales the scale warp loads in one burst
constexpr int kScSlots = 16;  // two bursts: one being consumed while the next is loaded
struct ScaleRing {
  float a[kScSlots][128];
  float b[kScSlots][4];
  uint64_t full[kScSlots];   // 32 arrivals: every lane of the scale warp after its stores
  uint64_t empty[kScSlots];  // one arrival per promoter warp after its reads
};
constexpr int kScaleRingBytes = (int)((sizeof(ScaleRing) + 127) / 128 * 128);
static_assert(sizeof(Shared) <= kSharedBytes, "shared block");

FP8_DEVI int find_expert(const int32_t* tpre, int E, int64_t t) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tpre[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Tile t of the persistent schedule. Tile indices, tile counts and block coordinates fit in 32
// bits (the launcher checks), so the divisions here are 32-bit: they sit on the MMA issuer's and
// the epilogue's per-tile path.
template <int SCHED, int TILE_M, int TBN>
FP8_DEVI Tile get_tile(const GemmParams& p, int64_t t64, const int32_t* tpre, const int32_t* aux,
                       const int32_t* pst) {
  Tile T;
  const uint32_t t = (uint32_t)t64, num_n = (uint32_t)p.num_n;
  if (is_dense(SCHED)) {
    uint32_t mb, nb;
    if (p.group_n == 0) {
      const uint32_t gm = (uint32_t)p.group_m;
      const uint32_t per_group = gm * num_n;
      const uint32_t g = t / per_group, r = t - g * per_group;
      const uint32_t first_m = g * gm;
      const uint32_t left = (uint32_t)p.num_m - first_m;
      const uint32_t gsz = left < gm ? left : gm;
      nb = r / gsz;
      mb = first_m + (r - nb * gsz);
    } else {
      const uint32_t gn = (uint32_t)p.group_n;
      const uint32_t per_group = gn * (uint32_t)p.num_m;
      const uint32_t g = t / per_group, r = t - g * per_group;
      const uint32_t first_n = g * gn;
      const uint32_t left = num_n - first_n;
      const uint32_t gsz = left < gn ? left : gn;
      mb = r / gsz;
      nb = first_n + (r - mb * gsz);
    }
    T.m0 = (int64_t)mb * TILE_M;
    T.pm0 = T.m0;
    T.n0 = (int64_t)nb * TBN;
    T.row_end = p.M;
    T.k0 = 0;
    T.nkb = p.nkb;
    T.e = 0;
    T.tt = 0;
  } else if (SCHED == kJagM) {
    const int e = find_expert(tpre, p.E, t64);
    const uint32_t local = t - (uint32_t)tpre[e];
    const uint32_t mb = local / num_n, nb = local - mb * num_n;
    T.m0 = aux[e] + (int64_t)mb * TILE_M;  // aux[e] = segment start row
    T.pm0 = pst ? pst[e] + (int64_t)mb * TILE_M : T.m0;
    T.n0 = (int64_t)nb * TBN;
    T.row_end = aux[e + 1];
    T.k0 = 0;
    T.nkb = p.nkb;
    T.e = e;
    T.tt = (p.tail_t && T.row_end - T.m0 < TILE_M) ? (int)(T.row_end - T.m0) : 0;
  } else {
    const uint32_t per = (uint32_t)p.num_m * num_n;
    const uint32_t e = t / per;
    const uint32_t local = t - e * per;
    const uint32_t mb = local / num_n, nb = local - mb * num_n;
    T.m0 = (int64_t)mb * TILE_M;
    T.pm0 = T.m0;
    T.n0 = (int64_t)nb * TBN;
    T.row_end = p.M;
    T.k0 = aux[e];                             // aux[e] = padded start of segment e
    T.nkb = (aux[e + 1] - aux[e]) / BKB;       // padded length / 128
    T.e = (int)e;
    T.tt = 0;
  }
  return T;
}

// K blocks of tile t (all the MMA issuer needs to know about a tile).
template <int SCHED>
FP8_DEVI int64_t tile_nkb(const GemmParams& p, int64_t t, const int32_t* aux) {
  if (SCHED != kJagK) return p.nkb;
  const uint32_t e = (uint32_t)t / ((uint32_t)p.num_m * (uint32_t)p.num_n);
  return (aux[e + 1] - aux[e]) / BKB;
}

template <int KIND, int SCHED, int A_MN, int B_MN, int CG>
__global__ void __launch_bounds__(Cfg<KIND, CG, SCHED>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmSA,
                const __grid_constant__ CUtensorMap tmSB, const GemmParams p) {
  using C = Cfg<KIND, CG, SCHED>;
  static_assert(C::STAGES <= kMaxStages && C::NBUF <= 4, "ring and accumulator barriers fit the shared block");
  constexpr int STAGES = C::STAGES;
  constexpr int kThreads = C::THREADS;
  constexpr int kEpiThreads = C::EPI_THREADS;
  constexpr int TBN = C::TBN;
  constexpr bool kPadRows = KIND == kMX && SCHED == kJagM;  // A scales in the segment-padded row space
  // FP8 jagged M on pairs: transposed tail tiles, whose row boxes of 32 and 64 rows come in the
  // tmSA and tmSB slots (unused by FP8 operands); 128-row boxes are tmA's own
  constexpr bool kTail = KIND == kFP8 && SCHED == kJagM && CG == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + C::RING_BYTES;  // [8 warps][kStageOut], pairs only
  Shared& S = *reinterpret_cast<Shared*>(smem + C::RING_BYTES + C::OUT_BYTES);
  int32_t* tpre = reinterpret_cast<int32_t*>(smem + C::RING_BYTES + C::OUT_BYTES + kSharedBytes);
  int32_t* aux = tpre + (p.E + 1);
  ScaleRing& SR = *reinterpret_cast<ScaleRing*>(smem + C::RING_BYTES + C::OUT_BYTES + kSharedBytes);  // kBLK (dense)
  int32_t* pst = kPadRows ? aux + (p.E + 1) : nullptr;  // padded segment starts
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &S.abort;
  const uint32_t rank = CG == 2 ? cluster_ctarank() : 0;  // 0 issues the pair's MMAs
  const bool issuer = rank == 0;
  const int64_t unit = blockIdx.x / CG, n_units = gridDim.x / CG;

  // ---- jagged schedules: validate offsets, per-expert tile prefix and row / K starts ----
  int64_t total;
  if (is_dense(SCHED)) {
    total = p.num_m * p.num_n;
  } else {
    int bad = 0;
    for (int e = tid; e < p.E; e += kThreads) {
      const int32_t cur = p.ends[e], prev = e ? p.ends[e - 1] : 0;
      if (cur < prev || (SCHED != kJagK && e == p.E - 1 && cur != p.total_rows)) bad = 1;
      const int64_t cnt = cur > prev ? cur - prev : 0;
      if (SCHED == kJagM) {
        tpre[e + 1] = (int32_t)(((cnt + C::TILE_M - 1) / C::TILE_M) * p.num_n);
        aux[e + 1] = cur;
        if (kPadRows) pst[e + 1] = (int32_t)((cnt + 127) / 128 * 128);
      } else {
        tpre[e + 1] = (int32_t)(p.num_m * p.num_n);
        aux[e + 1] = (int32_t)(((cnt + BKB - 1) / BKB) * BKB);
      }
    }
    if (tid == 0) {
      tpre[0] = 0;
      aux[0] = 0;
      if (kPadRows) pst[0] = 0;
    }
    bad = __syncthreads_or(bad);
    if (bad) {  // both CTAs of a pair see the same offsets and leave together
      if (blockIdx.x == 0 && tid == 0) set_status(p.status, FP8_DEV_BAD_OFFSETS);
      return;
    }
    if (warp == 0) {  // inclusive scans (tile prefix always; padded prefix for jagged K / MX rows)
      constexpr bool kScan2 = SCHED == kJagK || kPadRows;
      int32_t* w_arr = SCHED == kJagK ? aux : pst;
      int carry = 0, carry2 = 0;
      for (int base = 0; base < p.E; base += 32) {
        const int i = base + lane;
        int v = i < p.E ? tpre[i + 1] : 0;
        int w = (kScan2 && i < p.E) ? w_arr[i + 1] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, v, o);
          const int z = __shfl_up_sync(0xffffffffu, w, o);
          if (lane >= o) {
            v += y;
            w += z;
          }
        }
        if (i < p.E) {
          tpre[i + 1] = v + carry;
          if (kScan2) w_arr[i + 1] = w + carry2;
        }
        carry += __shfl_sync(0xffffffffu, v, 31);
        carry2 += __shfl_sync(0xffffffffu, w, 31);
      }
    }
    __syncthreads();
    total = tpre[p.E];
    if (SCHED == kJagK && aux[p.E] > p.K) {  // segments do not fit the padded operand
      if (blockIdx.x == 0 && tid == 0) set_status(p.status, FP8_DEV_BAD_OFFSETS);
      return;
    }
  }

  // ---- barriers and tensor memory ----
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(&S.tfull[b], 1);
      mbar_init(&S.tempty[b], CG * kEpiThreads / 32);
    }
    mbar_init(&S.drain, 1);
    for (int s2 = 0; s2 < STAGES; ++s2) mbar_init(&S.sff[s2], 1);
    mbar_init(&S.sf_drain, 1);
    if (KIND == kBLK) {
      for (int i = 0; i < kScSlots; ++i) {
        mbar_init(&SR.full[i], 32);
        mbar_init(&SR.empty[i], C::EPI_WARPS);
      }
    }
    mbar_init(&S.never, 1);
    S.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (CG == 2) tma_prefetch_desc(&tmO);
    if (KIND == kMX || (kTail && p.tail_t)) {
      tma_prefetch_desc(&tmSA);
      tma_prefetch_desc(&tmSB);
    }
  }
  if (warp == 1) {
    if (CG == 2) {
      tmem_alloc_pair(&S.tmem_base, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&S.tmem_base, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_barrier();  // the peer's barriers are initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = S.tmem_base;

  auto fail = [&]() {
    *abort_flag = 1;
    set_status(p.status, FP8_DEV_TIMEOUT);
  };

  if (warp == 0) {
    // ================================ TMA producer ================================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int64_t t = unit; t < total && ok; t += n_units) {
        const Tile T = get_tile<SCHED, C::TILE_M, TBN>(p, t, tpre, aux, pst);
        const int32_t am = (int32_t)(T.m0 + (int64_t)rank * BM);        // this CTA's A rows
        const int32_t bn = (int32_t)(T.n0 + (int64_t)rank * C::B_ROWS);  // this CTA's B rows
        // MX scale blocks: this CTA's 128 A rows; the two 128-row B blocks holding the tile's
        // columns (each CTA of a pair loads them in full: its accumulator spans all columns)
        const int32_t sfa_rb = (int32_t)((T.pm0 + (int64_t)rank * BM) / 128);
        const int32_t sfb_rb = (int32_t)(T.n0 / 128);
        // transposed tail tile: each CTA holds N' / 2 of its rows (N' = rows rounded up to 16),
        // loaded with the smallest row box that covers them; the weight rows take the A side
        int tail_half = 0, tail_box = 0;
        if (kTail && T.tt) {
          tail_half = (T.tt + 15) / 16 * 8;
          tail_box = tail_half <= 32 ? 32 : (tail_half <= 64 ? 64 : 128);
        }
        const uint32_t tx = tail_box ? (uint32_t)(C::A_BYTES + tail_box * BKB) : (uint32_t)C::TX_BYTES;
        for (int64_t kb = 0; kb < T.nkb; ++kb) {
          if (!mbar_wait(&S.empty[stage], phase ^ 1, abort_flag, p.wait_ns)) {
            if (!*abort_flag) fail();
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * C::STAGE_BYTES;
          uint8_t* sb = sa + C::A_BYTES;
          uint8_t* ssf = sa + C::A_BYTES + C::B_BYTES;
          if (CG == 1) {
            uint64_t* fb = &S.full[stage];
            mbar_arrive_expect_tx(fb, C::TX_BYTES);
            if (KIND == kMX) {
              const int32_t kx = (int32_t)(T.k0 + kb * BKB);
              tma_load_2d(sa, &tmA, fb, kx, am);
              if (SCHED == kJagM) {
                tma_load_3d(sb, &tmB, fb, kx, bn, T.e);
                tma_load_4d(ssf + 512, &tmSB, fb, 0, kx / 128, sfb_rb, T.e);
              } else {
                tma_load_2d(sb, &tmB, fb, kx, bn);
                tma_load_3d(ssf + 512, &tmSB, fb, 0, kx / 128, sfb_rb);
              }
              tma_load_3d(ssf, &tmSA, fb, 0, kx / 128, sfa_rb);
            } else if (KIND == kFP8 || KIND == kBLK) {
              const int32_t kx = (int32_t)(T.k0 + kb * BKB);
              tma_load_2d(sa, &tmA, fb, kx, am);
              if (SCHED == kJagM)
                tma_load_3d(sb, &tmB, fb, kx, bn, T.e);
              else
                tma_load_2d(sb, &tmB, fb, kx, bn);
            } else {
              const int32_t kx = (int32_t)(kb * (BKB / 2));  // 64 bf16 per block
              if (A_MN) {
                tma_load_2d(sa, &tmA, fb, am, kx);
                tma_load_2d(sa + 8192, &tmA, fb, am + 64, kx);
              } else {
                tma_load_2d(sa, &tmA, fb, kx, am);
              }
              if (B_MN) {
#pragma unroll
                for (int h = 0; h < C::B_ROWS / 64; ++h) tma_load_2d(sb + h * 8192, &tmB, fb, bn + 64 * h, kx);
              } else {
                tma_load_2d(sb, &tmB, fb, kx, bn);
              }
            }
          } else {
            // both CTAs' bytes are counted on the issuing CTA's full barrier
            const uint32_t fb = mapa_shared(smem_u32(&S.full[stage]), 0);
            if (issuer) mbar_arrive_expect_tx(&S.full[stage], 2 * tx);
            if (KIND == kMX) {
              const int32_t kx = (int32_t)(T.k0 + kb * BKB);
              tma_load_2d_pair(sa, &tmA, fb, kx, am);
              if (SCHED == kJagM) {
                tma_load_3d_pair(sb, &tmB, fb, kx, bn, T.e);
                tma_load_4d_pair(ssf + 512, &tmSB, fb, 0, kx / 128, sfb_rb, T.e);
              } else {
                tma_load_2d_pair(sb, &tmB, fb, kx, bn);
                tma_load_3d_pair(ssf + 512, &tmSB, fb, 0, kx / 128, sfb_rb);
              }
              tma_load_3d_pair(ssf, &tmSA, fb, 0, kx / 128, sfa_rb);
            } else if (KIND == kFP8 || KIND == kBLK) {
              const int32_t kx = (int32_t)(T.k0 + kb * BKB);
              if (kTail && tail_box) {
                tma_load_3d_pair(sa, &tmB, fb, kx, bn, T.e);  // this CTA's 128 weight rows
                const CUtensorMap* tm = tail_box == 32 ? &tmSA : (tail_box == 64 ? &tmSB : &tmA);
                tma_load_2d_pair(sb, tm, fb, kx, (int32_t)(T.m0 + (int64_t)rank * tail_half));
              } else {
                tma_load_2d_pair(sa, &tmA, fb, kx, am);
                if (SCHED == kJagM)
                  tma_load_3d_pair(sb, &tmB, fb, kx, bn, T.e);
                else
                  tma_load_2d_pair(sb, &tmB, fb, kx, bn);
              }
            } else {
              const int32_t kx = (int32_t)(kb * (BKB / 2));
              if (A_MN) {
                tma_load_2d_pair(sa, &tmA, fb, am, kx);
                tma_load_2d_pair(sa + 8192, &tmA, fb, am + 64, kx);
              } else {
                tma_load_2d_pair(sa, &tmA, fb, kx, am);
              }
              if (B_MN) {
#pragma unroll
                for (int h = 0; h < C::B_ROWS / 64; ++h) tma_load_2d_pair(sb + h * 8192, &tmB, fb, bn + 64 * h, kx);
              } else {
                tma_load_2d_pair(sb, &tmB, fb, kx, bn);
              }
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Drain: the last (up to STAGES) loads must land before the CTA (pair) may exit. For a
      // pair, the issuing CTA's full barriers count both CTAs' loads; after an abort the other
      // CTA cannot observe them and lets its own last loads settle for 100 us instead.
      if (issuer) {
        const int64_t first = issued > STAGES ? issued - STAGES : 0;
        for (int64_t i = first; i < issued; ++i)
          mbar_wait(&S.full[i % STAGES], (uint32_t)((i / STAGES) & 1), nullptr, kDrainNs);
      } else if (!ok) {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================================ MMA issuer ================================
    if (lane == 0 && issuer) {
      int stage = 0;
      uint32_t phase = 0;
      int buf = 0;
      uint32_t aphase = 0;
      bool ok = true;
      // MX: stage 0's A descriptor and the four scale-factor ids
      const uint64_t mx_a_desc0 = smem_desc(smem_u32(smem), 16, 1024);
      uint32_t mx_id[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) mx_id[kk] = idesc_sf_ids(p.idesc, (uint32_t)kk, (uint32_t)kk);
      if (p.test_stall && !mbar_wait(&S.never, 0, abort_flag, p.wait_ns)) {
        fail();
        ok = false;
      }
      for (int64_t t = unit; t < total && ok; t += n_units) {
        const int64_t nkb = tile_nkb<SCHED>(p, t, aux);
        if (nkb == 0) continue;
        uint32_t idesc = p.idesc;
        if (kTail && p.tail_t) {  // transposed tail tile: swapped formats, N = N'
          const int tt = get_tile<SCHED, C::TILE_M, TBN>(p, t, tpre, aux, pst).tt;
          if (tt) idesc = p.idesc_t | ((uint32_t)((tt + 15) / 16 * 2) << 17);
        }
        if (KIND != kBLK) {
          if (!mbar_wait(&S.tempty[buf], aphase ^ 1, abort_flag, p.wait_ns)) {
            if (!*abort_flag) fail();
            break;
          }
          tc_fence_after();
        }
        uint32_t d_tmem = tmem_base + (uint32_t)(buf * TBN);
        for (int64_t kb = 0; kb < nkb; ++kb) {
          if (KIND == kBLK) {  // each K block into the next free partial buffer
            if (!mbar_wait(&S.tempty[buf], aphase ^ 1, abort_flag, p.wait_ns)) {
              if (!*abort_flag) fail();
              ok = false;
              break;
            }
            tc_fence_after();
            d_tmem = tmem_base + (uint32_t)(buf * TBN);
          }
          // MX: the scale warp's commit on sff[stage] follows the stage's full barrier
          if (!mbar_wait(KIND == kMX ? &S.sff[stage] : &S.full[stage], phase, abort_flag, p.wait_ns)) {
            if (!*abort_flag) fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
          if (KIND == kMX) {
            // the stage's scales are in its tensor-memory slot (copied by the scale warp).
            // Descriptors are offsets of per-kernel bases (address field in 16-byte units), so
            // the single issuing thread spends few instructions per stage.
            const uint32_t sf_t = tmem_base + (uint32_t)(C::SF_COL0 + 16 * stage);
            const uint64_t soff = (uint64_t)((stage * C::STAGE_BYTES) >> 4);
            const uint64_t ad0 = mx_a_desc0 + soff;
            const uint32_t sfb_t = sf_t + 4;  // 256-column tiles start on a 128-row scale block
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = ad0 + 2 * kk;
              const uint64_t bd = ad + (C::A_BYTES >> 4);
              const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
              if (CG == 2)
                umma_mx_pair(d_tmem, ad, bd, mx_id[kk], sf_t, sfb_t, acc);
              else
                umma_mx(d_tmem, ad, bd, mx_id[kk], sf_t, sfb_t, acc);
            }
          } else {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = A_MN ? smem_desc(sa + kk * 2048, 8192, 1024) : smem_desc(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc(sb + kk * 2048, 8192, 1024) : smem_desc(sb + kk * 32, 16, 1024);
            const uint32_t acc = ((KIND != kBLK && kb > 0) || kk > 0) ? 1u : 0u;
            if (CG == 2) {
              if (KIND == kFP8 || KIND == kBLK)
                umma_f8f6f4_pair(d_tmem, ad, bd, idesc, acc);
              else
                umma_f16_pair(d_tmem, ad, bd, p.idesc, acc);
            } else {
              if (KIND == kFP8 || KIND == kBLK)
                umma_f8f6f4(d_tmem, ad, bd, p.idesc, acc);
              else
                umma_f16(d_tmem, ad, bd, p.idesc, acc);
            }
          }
          }
          // frees the stage (in both CTAs of a pair) once these MMAs have read it
          if (CG == 2)
            umma_commit_pair(&S.empty[stage], 0x3);
          else
            umma_commit(&S.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (KIND == kBLK) {  // this K block's partial is ready for promotion
            if (CG == 2)
              umma_commit_pair(&S.tfull[buf], 0x3);
            else
              umma_commit(&S.tfull[buf]);
            if (++buf == C::NBUF) {
              buf = 0;
              aphase ^= 1;
            }
          }
        }
        if (!ok) break;
        if (KIND == kBLK) continue;
        // accumulator ready for the epilogue(s)
        if (CG == 2)
          umma_commit_pair(&S.tfull[buf], 0x3);
        else
          umma_commit(&S.tfull[buf]);
        if (++buf == C::NBUF) {
          buf = 0;
          aphase ^= 1;
        }
      }
      // Drain every MMA this thread issued before the tensor memory is released.
      if (CG == 2)
        umma_commit_pair(&S.drain, 0x3);
      else
        umma_commit(&S.drain);
    }
    __syncwarp();
  } else if (KIND == kBLK && warp == C::SF_WARP) {
    // ======================= blockwise: tile scales, K block by K block =======================
    // For every K block of every tile this CTA computes: this CTA's 128 row scales
    // sA[m, kb] (lane l holds rows l, l + 32, l + 64, l + 96) and the two 128-column block
    // scales sB[n / 128, kb], into the next ring slot. The loads for kScGroup K blocks go out
    // together (one memory latency per burst, not per block), and the ring holds two bursts.
    int slot = 0;
    uint32_t ph = 0;
    const int64_t KB = p.nkb;
    bool ok = true;
    for (int64_t t = unit; t < total && ok; t += n_units) {
      const Tile T = get_tile<SCHED, C::TILE_M, TBN>(p, t, tpre, aux, pst);
      const int64_t r0 = T.m0 + (int64_t)rank * BM;
      const int64_t nb = T.n0 / 128 + (lane & 1);
      const bool b_live = lane < 2 && nb * 128 < p.N;
      for (int64_t kb0 = 0; kb0 < T.nkb && ok; kb0 += kScGroup) {
        float va[4][kScGroup], vb[kScGroup];
#pragma unroll
        for (int j = 0; j < kScGroup; ++j) {
          const bool k_live = kb0 + j < T.nkb;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int64_t r = r0 + lane + 32 * i;
            va[i][j] = (k_live && r < p.M) ? __ldg(p.sA + r * KB + kb0 + j) : 0.0f;
          }
          vb[j] = (k_live && b_live) ? __ldg(p.sB + nb * KB + kb0 + j) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kScGroup; ++j) {
          if (kb0 + j >= T.nkb) break;
          if (!mbar_wait(&SR.empty[slot], ph ^ 1, abort_flag, p.wait_ns)) {
            if (!*abort_flag) fail();
            ok = false;
            break;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) SR.a[slot][lane + 32 * i] = va[i][j];
          if (lane < 2) SR.b[slot][lane] = vb[j];
          mbar_arrive(&SR.full[slot]);  // release: this lane's stores before the arrival
          if (++slot == kScSlots) {
            slot = 0;
            ph ^= 1;
          }
        }
      }
    }
    __syncwarp();
  } else if (KIND == kMX && warp == C::SF_WARP) {
    // ============================ MX scale copies ============================
    // For every stage the MMA thread will consume: wait for its loads, copy its three scale
    // blocks into the stage's tensor-memory slot (shared memory -> tensor memory), and commit
    // them to sff[stage]. Issued apart from the MMAs so that a copy never waits behind them;
    // the slot is free because the stage was refilled only after its previous MMAs completed.
    if (lane == 0 && issuer) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint64_t cp_desc0 = smem_desc_plain(smem_u32(smem) + C::A_BYTES + C::B_BYTES, 128);
      for (int64_t t = unit; t < total && ok; t += n_units) {
        const int64_t nkb = tile_nkb<SCHED>(p, t, aux);
        for (int64_t kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&S.full[stage], phase, abort_flag, p.wait_ns)) {
            if (!*abort_flag) fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf_t = tmem_base + (uint32_t)(C::SF_COL0 + 16 * stage);
          const uint64_t cd = cp_desc0 + (uint64_t)((stage * C::STAGE_BYTES) >> 4);
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            if (CG == 2)
              tmem_cp_sf_pair(sf_t + 4 * j, cd + 32 * j);
            else
              tmem_cp_sf(sf_t + 4 * j, cd + 32 * j);
          }
          if (CG == 2)
            umma_commit_pair(&S.sff[stage], 0x1);
          else
            umma_commit(&S.sff[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // every copy into either CTA's tensor memory completes before it is released
      if (CG == 2)
        umma_commit_pair(&S.sf_drain, 0x3);
      else
        umma_commit(&S.sf_drain);
    }
    __syncwarp();
  } else {
    // ================================ epilogue ================================
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int c0 = ((warp - 2) >> 2) * C::WCOLS;  // first tile column of this warp's share
    const int etid = tid - 64;           // 0..255 across the epilogue warps
    const int row = (int)rank * BM + q * 32 + lane;  // row within the pair's tile
    const bool stage_sb = KIND == kFP8 && !p.sb_scalar;
    int buf = 0, sbi = 0;
    int sc_slot = 0;       // kBLK: scale-ring slot and phase
    uint32_t sc_ph = 0;
    uint32_t oseq = 0;  // TMA stores issued by this warp
    uint32_t aphase = 0;
    // The next tile and the scales it needs (this thread's row scale; its column scale, or the
    // scalar one) are fetched one tile ahead, so the memory latency hides behind this tile.
    Tile Tn;
    float sa_nx = 1.0f, sb_nx = 1.0f;
    auto fetch = [&](int64_t tt) {
      Tn = get_tile<SCHED, C::TILE_M, TBN>(p, tt, tpre, aux, pst);
      if (KIND != kFP8) return;
      if (kTail && Tn.tt) {  // this thread's weight-row scale; the staged scales are the rows'
        const int64_t n = Tn.n0 + row;
        sa_nx = n < p.N ? __ldg(p.sB + (int64_t)Tn.e * p.N + n) : 0.0f;
        sb_nx = etid < Tn.tt ? (p.sa_scalar ? __ldg(p.sA) : __ldg(p.sA + Tn.m0 + etid)) : 0.0f;
        return;
      }
      const int64_t m = Tn.m0 + row;
      const float* sbp = p.sB;
      if (!is_dense(SCHED)) sbp += (int64_t)Tn.e * p.N;
      sa_nx = 1.0f;
      if (m < Tn.row_end) {
        if (SCHED == kJagK)
          sa_nx = __ldg(p.sA + (int64_t)Tn.e * p.M + m);
        else
          sa_nx = p.sa_scalar ? __ldg(p.sA) : __ldg(p.sA + m);
      }
      if (stage_sb) {
        const int64_t n = Tn.n0 + etid;
        sb_nx = n < p.N ? __ldg(sbp + n) : 0.0f;
      } else {
        sb_nx = __ldg(sbp);
      }
    };
    if (unit < total) fetch(unit);
    for (int64_t t = unit; t < total; t += n_units) {
      const Tile T = Tn;
      const float sa = sa_nx, sb_mine = sb_nx;
      if (t + n_units < total) fetch(t + n_units);
      const int64_t m = T.m0 + row;
      const bool row_ok = m < T.row_end;
      const int64_t orow = SCHED == kJagK ? (int64_t)T.e * p.M + m : m;
      if (stage_sb || (kTail && T.tt)) {  // one column scale per epilogue thread; reused by all 128 rows
        S.sb[sbi][etid] = sb_mine;
        named_bar_sync(1, kEpiThreads);
      }
      const float* sbs = S.sb[sbi];
      sbi ^= 1;
      if (T.nkb == 0) {  // empty segment (jagged K): the result is zero
        if (row_ok) {
          for (int64_t n = T.n0 + c0; n < T.n0 + c0 + C::WCOLS && n < p.N; ++n) {
            if (p.out_f32)
              static_cast<float*>(p.out)[orow * p.ldo + n] = 0.0f;
            else
              static_cast<uint16_t*>(p.out)[orow * p.ldo + n] = 0;
          }
        }
        continue;
      }
      if (KIND == kBLK) {
        // promotion: for every K block, this warp's columns of the partial into registers, the
        // partial back to the MMAs, then acc += partial * sA[m, kb] * sB[n / 128, kb] (the
        // warp's columns lie in one 128-column scale block). Stores after the last block.
        constexpr int WC = C::WCOLS, NL = WC / 16;
        const int bsel = c0 / 128;  // which of the tile's two 128-column scale blocks
        float acc[WC];
#pragma unroll
        for (int j = 0; j < WC; ++j) acc[j] = 0.0f;
        const uint32_t tq = ((uint32_t)(q * 32) << 16) + (uint32_t)c0;
        bool live = true;
        for (int64_t kb = 0; kb < T.nkb; ++kb) {
          // this K block's scales from the ring (staged ahead by the scale warp)
          if (!mbar_wait(&SR.full[sc_slot], sc_ph, abort_flag, p.wait_ns)) {
            if (!*abort_flag) fail();
            live = false;
            break;
          }
          const float sk = SR.a[sc_slot][q * 32 + lane] * SR.b[sc_slot][bsel];
          __syncwarp();
          if (lane == 0) mbar_arrive(&SR.empty[sc_slot]);
          if (++sc_slot == kScSlots) {
            sc_slot = 0;
            sc_ph ^= 1;
          }
          if (!mbar_wait(&S.tfull[buf], aphase, abort_flag, p.wait_ns)) {
            if (!*abort_flag) fail();
            live = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + (uint32_t)(buf * TBN) + tq;
          // 16 columns at a time (the accumulators already hold WC registers); overlapping the
          // loads with the adds through a second staging set measured no faster
          uint32_t v[16];
#pragma unroll
          for (int h = 0; h + 1 < NL; ++h) {
            tmem_ld16(taddr + 16 * h, v);
            tmem_ld_wait_regs16(v);
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[16 * h + j] = fmaf(__uint_as_float(v[j]), sk, acc[16 * h + j]);
          }
          tmem_ld16(taddr + 16 * (NL - 1), v);
          tmem_ld_wait_regs16(v);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (CG == 2)
              mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&S.tempty[buf]), 0));
            else
              mbar_arrive_relaxed(&S.tempty[buf]);
          }
          if (++buf == C::NBUF) {
            buf = 0;
            aphase ^= 1;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[16 * (NL - 1) + j] = fmaf(__uint_as_float(v[j]), sk, acc[16 * (NL - 1) + j]);
        }
        if (!live) break;
        if (row_ok) {
#pragma unroll
          for (int h = 0; h < WC / 32; ++h) {
            const int64_t n = T.n0 + c0 + 32 * h;
            if (n >= p.N) break;
            const float* a = acc + 32 * h;
            const bool full = p.vec_ok && n + 32 <= p.N;
            if (p.out_f32) {
              float* o = static_cast<float*>(p.out) + orow * p.ldo + n;
              if (full) {
#pragma unroll
                for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(o + j) = make_float4(a[j], a[j + 1], a[j + 2], a[j + 3]);
              } else {
                for (int j = 0; j < 32 && n + j < p.N; ++j) o[j] = a[j];
              }
            } else {
              uint16_t* o = static_cast<uint16_t*>(p.out) + orow * p.ldo + n;
              uint32_t wd[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const __nv_bfloat162 hb = __floats2bfloat162_rn(a[2 * j], a[2 * j + 1]);
                wd[j] = *reinterpret_cast<const uint32_t*>(&hb);
              }
              if (full) {
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                  *reinterpret_cast<uint4*>(o + 2 * j) = make_uint4(wd[j], wd[j + 1], wd[j + 2], wd[j + 3]);
              } else {
                for (int j = 0; j < 32 && n + j < p.N; ++j) o[j] = (uint16_t)(wd[j >> 1] >> (16 * (j & 1)));
              }
            }
          }
        }
        continue;
      }
      const bool got = mbar_wait(&S.tfull[buf], aphase, abort_flag, p.wait_ns);
      if (!named_bar_and(2, kEpiThreads, got)) {  // uniform decision across the epilogue warps
        if (!got && !*abort_flag) fail();
        break;
      }
      tc_fence_after();
      if (KIND == kMX) {
        // this warp's 64 columns into registers, the accumulator back to the MMAs, then stores
        const uint32_t taddr = tmem_base + (uint32_t)c0 + ((uint32_t)(q * 32) << 16);
        uint32_t va[32], vb[32];
        tmem_ld32(taddr, va);
        tmem_ld32(taddr + 32, vb);
        tmem_ld_wait_regs(va);
        tmem_ld_wait_regs(vb);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (CG == 2)
            mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&S.tempty[0]), 0));
          else
            mbar_arrive_relaxed(&S.tempty[0]);
        }
        aphase ^= 1;
        if (C::MX_TMA_OUT && p.tma_out && !p.out_f32 && T.n0 + c0 < p.N) {
          // jagged K: bf16 through a 128-byte-swizzled [32 rows][128 B] box and one TMA store
          // per warp and tile (columns past N are clipped by the copy)
          const int64_t wrow0 = T.m0 + (int64_t)rank * BM + q * 32;
          uint8_t* st = out_stage + (warp - 2) * kStageOut;
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const __nv_bfloat162 h0 = __floats2bfloat162_rn(__uint_as_float(va[2 * j]), __uint_as_float(va[2 * j + 1]));
            const __nv_bfloat162 h1 = __floats2bfloat162_rn(__uint_as_float(vb[2 * j]), __uint_as_float(vb[2 * j + 1]));
            w[j] = *reinterpret_cast<const uint32_t*>(&h0);
            w[16 + j] = *reinterpret_cast<const uint32_t*>(&h1);
          }
          if (lane == 0) bulk_wait_read_all();  // the previous tile's store has read the buffer
          __syncwarp();
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8)
            *reinterpret_cast<uint4*>(st + lane * 128 + ((c8 ^ (lane & 7)) << 4)) =
                make_uint4(w[4 * c8], w[4 * c8 + 1], w[4 * c8 + 2], w[4 * c8 + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmO, st, (int32_t)(T.n0 + c0), (int32_t)wrow0, T.e);
            bulk_commit();
          }
          continue;
        }
        if (row_ok) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t* v = h ? vb : va;
            const int64_t n = T.n0 + c0 + 32 * h;
            if (n >= p.N) break;
            const bool full = p.vec_ok && n + 32 <= p.N;
            if (p.out_f32) {
              float* o = static_cast<float*>(p.out) + orow * p.ldo + n;
              if (full) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                  *reinterpret_cast<uint4*>(o + j) = make_uint4(v[j], v[j + 1], v[j + 2], v[j + 3]);
              } else {
                for (int j = 0; j < 32 && n + j < p.N; ++j) o[j] = __uint_as_float(v[j]);
              }
            } else {
              uint16_t* o = static_cast<uint16_t*>(p.out) + orow * p.ldo + n;
              uint32_t wd[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const __nv_bfloat162 hb = __floats2bfloat162_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                wd[j] = *reinterpret_cast<const uint32_t*>(&hb);
              }
              if (full) {
#pragma unroll
                for (int j = 0; j < 16; j += 4)
                  *reinterpret_cast<uint4*>(o + 2 * j) = make_uint4(wd[j], wd[j + 1], wd[j + 2], wd[j + 3]);
              } else {
                for (int j = 0; j < 32 && n + j < p.N; ++j) o[j] = (uint16_t)(wd[j >> 1] >> (16 * (j & 1)));
              }
            }
          }
        }
        continue;
      }
      const float sb_all = (KIND == kFP8 && p.sb_scalar) ? sb_mine : 1.0f;
      const uint32_t taddr = tmem_base + (uint32_t)(buf * TBN + c0) + ((uint32_t)(q * 32) << 16);
      if (kTail && T.tt) {
        // transposed tail tile: lane = weight row n (an output column), tensor-memory column j =
        // the tile's row m0 + j. Rounded as the ordinary tiles round, (acc * sA[m]) * sB[n]. For
        // each row the warp's lanes hold 32 consecutive output columns: every store instruction
        // writes 64 (bf16) or 128 (fp32) contiguous bytes; rows past the tile's end are skipped.
        const int64_t n = T.n0 + row;
        const bool n_ok = n < p.N;
        const float2 sn2 = make_float2(sa, sa);
        uint32_t v[32];
        for (int ch = 0; ch < C::WCOLS / 32; ++ch) {
          const int cl = c0 + ch * 32;
          if (cl >= T.tt) break;  // uniform across the warp
          tmem_ld32(taddr + ch * 32, v);
          tmem_ld_wait_regs(v);
          const int nr = T.tt - cl < 32 ? T.tt - cl : 32;
          const int64_t o0 = (T.m0 + cl) * p.ldo + n;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 x = fmul2_rn(fmul2_rn(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])),
                                               *reinterpret_cast<const float2*>(sbs + cl + j)),
                                      sn2);
            if (n_ok && j < nr) {
              if (p.out_f32) {
                float* o = static_cast<float*>(p.out) + o0 + j * p.ldo;
                o[0] = x.x;
                if (j + 1 < nr) o[p.ldo] = x.y;
              } else {
                __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + o0 + j * p.ldo;
                o[0] = __float2bfloat16_rn(x.x);
                if (j + 1 < nr) o[p.ldo] = __float2bfloat16_rn(x.y);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&S.tempty[buf]), 0));
        if (++buf == 2) {
          buf = 0;
          aphase ^= 1;
        }
        continue;
      }
      if constexpr (SCHED == kDenseQuant) {
        // The next quantization from the epilogue ("Triton Kernel Optimization", Level 1): this
        // lane holds row m's tile columns c0 .. c0 + 127. They are scaled and rounded once to bf16
        // (the result as fp8_scaled_mm stores it), the accumulator goes back to the MMAs, and the
        // bf16 values are quantized along the row: one 1 x 128 block (scale by the recipe's table)
        // or four MX blocks of 32 (E8M0 scales). Codes leave as the row's 128 bytes; the scales
        // beside them.
        static_assert(C::WCOLS == 128, "one 128-column row segment per lane");
        uint32_t h[64];
        const float2 sa2 = make_float2(sa, sa);
        uint32_t v[32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          tmem_ld32(taddr + ch * 32, v);
          tmem_ld_wait_regs(v);
          const int cl = c0 + ch * 32;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 sb2 = stage_sb ? *reinterpret_cast<const float2*>(sbs + cl + j) : make_float2(sb_all, sb_all);
            const float2 x = fmul2_rn(fmul2_rn(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), sa2), sb2);
            const __nv_bfloat162 hb = __floats2bfloat162_rn(x.x, x.y);
            h[ch * 16 + j / 2] = *reinterpret_cast<const uint32_t*>(&hb);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (CG == 2)
            mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&S.tempty[buf]), 0));
          else
            mbar_arrive_relaxed(&S.tempty[buf]);
        }
        if (++buf == 2) {
          buf = 0;
          aphase ^= 1;
        }
        const int64_t n0 = T.n0 + c0;
        if (!row_ok || n0 >= p.N) continue;  // N % 128 == 0: the segment is all in range or all out
        const bool e4 = p.q_fmt == FP8_DT_E4M3;
        uint32_t qw[32];
        if (p.q_mx) {
          uint32_t codes = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t am = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) am = absmax2(am, h[16 * b + j]);
            const uint32_t code = e4 ? mx_code<FP8_DT_E4M3>(absmax_fold(am)) : mx_code<FP8_DT_E5M2>(absmax_fold(am));
            const float inv = mx_inv(code);
            codes |= code << (8 * b);
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              const uint32_t lo = e4 ? mx_cast2<FP8_DT_E4M3>(h[16 * b + j], inv) : mx_cast2<FP8_DT_E5M2>(h[16 * b + j], inv);
              const uint32_t hi = e4 ? mx_cast2<FP8_DT_E4M3>(h[16 * b + j + 1], inv) : mx_cast2<FP8_DT_E5M2>(h[16 * b + j + 1], inv);
              qw[8 * b + j / 2] = lo | (hi << 16);
            }
          }
          // row m's four block codes: one aligned word of the MX scale layout (rows M, contraction N)
          const int64_t off = ((m / 128) * (p.N / 128) + n0 / 128) * 512 + (m % 32) * 16 + ((m / 32) % 4) * 4;
          *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.q_scales) + off) = codes;
        } else {
          uint32_t am = 0;
#pragma unroll
          for (int j = 0; j < 64; ++j) am = absmax2(am, h[j]);
          const Scale sc = tab_scale(p.q_tab, absmax_fold(am));
          const float2 s2 = make_float2(sc.s32, sc.s32);
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float2 a = fmul2_rn(make_float2(__uint_as_float(h[j] << 16), __uint_as_float(h[j] & 0xFFFF0000u)), s2);
            const float2 b = fmul2_rn(make_float2(__uint_as_float(h[j + 1] << 16), __uint_as_float(h[j + 1] & 0xFFFF0000u)), s2);
            const uint32_t lo = e4 ? cvt_fp8x2<FP8_DT_E4M3>(a.x, a.y) : cvt_fp8x2<FP8_DT_E5M2>(a.x, a.y);
            const uint32_t hi = e4 ? cvt_fp8x2<FP8_DT_E4M3>(b.x, b.y) : cvt_fp8x2<FP8_DT_E5M2>(b.x, b.y);
            qw[j / 2] = lo | (hi << 16);
          }
          static_cast<float*>(p.q_scales)[m * (p.N / 128) + n0 / 128] = sc.inv32;
        }
        uint4* dst = reinterpret_cast<uint4*>(p.q_out + m * p.N + n0);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_uint4(qw[4 * i], qw[4 * i + 1], qw[4 * i + 2], qw[4 * i + 3]);
        continue;
      }
      // Pairs write through shared memory with TMA bulk-tensor stores of 32 rows x 128 bytes
      // (64 bf16 columns, or 32 fp32), unless this warp's 32 rows run past the end of an
      // expert's segment.
      const int64_t wrow0 = T.m0 + (int64_t)rank * BM + q * 32;
      const bool via_tma = CG == 2 && p.tma_out && (SCHED != kJagM || wrow0 + 32 <= T.row_end);
      uint8_t* st = out_stage + (warp - 2) * kStageOut;
      // Two register sets: the load of the next 32 columns is in flight while the current ones
      // are scaled and stored (tcgen05.wait::ld names the set it completes, so the compiler
      // keeps that set in place until then).
      uint32_t va[32], vb[32];
      uint32_t w[32];  // bf16 pairs of two consecutive 32-column chunks (one 128-byte row)
      // Side outputs (dense schedule with amax): the maxima of |out| as stored (bf16), per row over
      // this warp's columns (one relaxed atomic max per row and tile) and per column over this
      // warp's 32 rows. Magnitudes of non-negative values order like their bit patterns, so all
      // maxima are integer maxima on packed pairs (vmax2). The column maxima of a 32 x 32 chunk
      // come from a butterfly across the lanes: each step keeps half of the words and folds in
      // the partner lane's other half (16 shuffles per chunk); the lanes then hold one column
      // pair each. Rows past the tile's end and columns past N count as zero.
      uint32_t racc = 0;
      auto amax_chunk = [&](const uint32_t* wv, int64_t n) {
        const int64_t left = p.N - n;
        const int valid = left >= 32 ? 32 : (left > 0 ? (int)left : 0);
        uint32_t m[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t v = wv[i] & 0x7FFF7FFFu;
          if (!row_ok || 2 * i >= valid) v = 0;
          else if (2 * i + 1 >= valid) v &= 0xFFFFu;
          m[i] = v;
          racc = __vmaxu2(racc, v);
        }
        if (!p.col_amax) return;
        // step with distance d (16, 8, 4, 2): the lanes with bit d clear keep words [0, h), the
        // others [h, 2h), each folding in the partner's copy of its kept half
#pragma unroll
        for (int h = 8; h >= 1; h >>= 1) {
          const int d = 2 * h;
          const bool upper = (lane & d) != 0;
#pragma unroll
          for (int i = 0; i < h; ++i) {
            const uint32_t keep = upper ? m[i + h] : m[i];
            const uint32_t give = upper ? m[i] : m[i + h];
            m[i] = __vmaxu2(keep, __shfl_xor_sync(0xffffffffu, give, d));
          }
        }
        m[0] = __vmaxu2(m[0], __shfl_xor_sync(0xffffffffu, m[0], 1));
        // the step of distance 2^k kept word bit (k - 1) from lane bit k, so lane l now holds the
        // column pair of word l >> 1; the even lane reports its low column, the odd one its high
        const int col = 2 * (lane >> 1) + (lane & 1);
        const uint32_t mc = (lane & 1) ? (m[0] >> 16) : (m[0] & 0xFFFFu);
        if (p.amax_whole) {
          const uint32_t mw = __reduce_max_sync(0xffffffffu, mc);
          if (lane == 0 && mw) red_max_relaxed(p.col_amax, mw << 16);
        } else if (col < valid && mc) {
          red_max_relaxed(p.col_amax + n + col, mc << 16);
        }
      };
      tmem_ld32(taddr, va);
      constexpr int NCH = C::WCOLS / 32;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) {
        uint32_t* v = (ch & 1) ? vb : va;
        tmem_ld_wait_regs(v);
        if (ch + 1 < NCH) tmem_ld32(taddr + (ch + 1) * 32, (ch & 1) ? va : vb);
        const int cl = c0 + ch * 32;  // tile column of v[0]
        const int64_t n = T.n0 + cl;
        // bf16 through TMA: the pair (ch - 1, ch) is stored once ch is done, unless the pair
        // starts at or past N (uniform across the warp); columns past N are clipped by the copy
        const bool pair_live = T.n0 + c0 + (ch & ~1) * 32 < p.N;
        if (n >= p.N && !(via_tma && !p.out_f32 && pair_live)) continue;
        float f[32];
        if (KIND == kMX) {  // the block scales were applied inside the MMA
#pragma unroll
          for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
        } else {
          const float2 sa2 = make_float2(sa, sa);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 sb2 = stage_sb ? *reinterpret_cast<const float2*>(sbs + cl + j) : make_float2(sb_all, sb_all);
            const float2 x = fmul2_rn(fmul2_rn(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), sa2), sb2);
            f[j] = x.x;
            f[j + 1] = x.y;
          }
        }
        if (via_tma) {
          if (!p.out_f32) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
              w[(ch & 1) * 16 + j] = *reinterpret_cast<const uint32_t*>(&h);
            }
            if (SCHED == kDenseAmax) amax_chunk(w + (ch & 1) * 16, n);
            if ((ch & 1) == 0) continue;
            if (lane == 0 && oseq >= 1) bulk_wait_read_all();  // the previous store has read the buffer
            __syncwarp();
            // row `lane` of a [32][128 B] box, 128-byte swizzle (16-byte chunk ^ row % 8)
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
              *reinterpret_cast<uint4*>(st + lane * 128 + ((c8 ^ (lane & 7)) << 4)) =
                  make_uint4(w[4 * c8], w[4 * c8 + 1], w[4 * c8 + 2], w[4 * c8 + 3]);
          } else {
            if (lane == 0 && oseq >= 1) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
              *reinterpret_cast<float4*>(st + lane * 128 + ((c8 ^ (lane & 7)) << 4)) =
                  make_float4(f[4 * c8], f[4 * c8 + 1], f[4 * c8 + 2], f[4 * c8 + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int32_t n_st = (int32_t)(p.out_f32 ? n : n - 32);
            if (SCHED == kJagK)
              tma_store_3d(&tmO, st, n_st, (int32_t)wrow0, T.e);
            else
              tma_store_2d(&tmO, st, n_st, (int32_t)wrow0);
            bulk_commit();
          }
          ++oseq;
          continue;
        }
        uint32_t wd[16];
        if (!p.out_f32) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
            wd[j] = *reinterpret_cast<const uint32_t*>(&h);
          }
          if (SCHED == kDenseAmax) amax_chunk(wd, n);
        }
        if (row_ok) {
          const bool full = p.vec_ok && n + 32 <= p.N;
          if (p.out_f32) {
            float* o = static_cast<float*>(p.out) + orow * p.ldo + n;
            if (full) {
#pragma unroll
              for (int j = 0; j < 32; j += 4) *reinterpret_cast<float4*>(o + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
            } else {
              for (int j = 0; j < 32 && n + j < p.N; ++j) o[j] = f[j];
            }
          } else {
            uint16_t* o = static_cast<uint16_t*>(p.out) + orow * p.ldo + n;
            if (full) {
#pragma unroll
              for (int j = 0; j < 16; j += 4) *reinterpret_cast<uint4*>(o + 2 * j) = make_uint4(wd[j], wd[j + 1], wd[j + 2], wd[j + 3]);
            } else {
              for (int j = 0; j < 32 && n + j < p.N; ++j) o[j] = (uint16_t)(wd[j >> 1] >> (16 * (j & 1)));
            }
          }
        }
      }
      if (SCHED == kDenseAmax && p.row_amax && row_ok) {
        const uint32_t r = (racc & 0xFFFFu) > (racc >> 16) ? (racc & 0xFFFFu) : (racc >> 16);
        if (r) red_max_relaxed(p.row_amax + orow, r << 16);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // the issuing CTA's barrier counts the epilogue warps of both CTAs
        if (CG == 2)
          mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&S.tempty[buf]), 0));
        else
          mbar_arrive_relaxed(&S.tempty[buf]);
      }
      if (++buf == 2) {
        buf = 0;
        aphase ^= 1;
      }
    }
  }

  if (CG == 2 && warp >= 2 && warp < 2 + C::EPI_WARPS && lane == 0) bulk_wait_all();  // this warp's stores are done
  tc_fence_before();
  __syncthreads();
  if (CG == 2) cluster_barrier();  // no remote arrive or load into a CTA that has left
  if (warp == 1) {
    if (lane == 0) {
      mbar_wait(&S.drain, 0, nullptr, kDrainNs);  // the MMAs writing this CTA's TMEM
      if (KIND == kMX) mbar_wait(&S.sf_drain, 0, nullptr, kDrainNs);  // and the scale copies
    }
    __syncwarp();
    tc_fence_after();
    if (CG == 2)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int KIND, int SCHED, int A_MN, int B_MN, int CG>
int run(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& o, const CUtensorMap& sfa,
        const CUtensorMap& sfb, const GemmParams& p, int64_t total_tiles_hint, const Ctx& c) {
  auto kern = gemm_kernel<KIND, SCHED, A_MN, B_MN, CG>;
  using C = Cfg<KIND, CG, SCHED>;
  constexpr int kThreads = C::THREADS;
  const int n_arrays = is_dense(SCHED) ? 0 : (KIND == kMX && SCHED == kJagM) ? 3 : 2;
  const size_t smem = 1024 + C::RING_BYTES + C::OUT_BYTES + kSharedBytes + (size_t)n_arrays * 4 * (p.E + 1) +
                     (KIND == kBLK ? kScaleRingBytes : 0);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return FP8_ERR_CUDA;
  int64_t units = c.sm_count / CG;
  if (total_tiles_hint > 0 && total_tiles_hint < units) units = total_tiles_hint;
  if (units < 1) units = 1;
  if (CG == 1) {
    kern<<<(unsigned)units, kThreads, smem, c.stream>>>(a, b, o, sfa, sfb, p);
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(units * CG));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, a, b, o, sfa, sfb, p) != cudaSuccess) return FP8_ERR_CUDA;
  return FP8_OK;
}

// MX operands: the FP8 codes load as on the FP8 path; the E8M0 scales, stored as
// [row blocks][K / 128][512 bytes], load through tensor maps over 128-word rows: a 3-D map
// [row block][K group][128 words] (4-D with the expert for the grouped weights). Box: one A
// block, two consecutive B blocks (a 192-column tile spans parts of at most two).
int launch_mx(const GemmArgs& g, GemmParams& p, const CUtensorMap& to, bool pair, int tile_m, const Ctx& c) {
  if (g.K % 128 || !g.sfa || !g.sfb) return FP8_ERR_UNSUPPORTED;
  const uint32_t af = g.a_dtype == FP8_DT_E4M3 ? kFmtE4M3 : kFmtE5M2;
  const uint32_t bf = g.b_dtype == FP8_DT_E4M3 ? kFmtE4M3 : kFmtE5M2;
  constexpr int TBN = Cfg<kMX, 1>::TBN;
  p.idesc = make_idesc_mx(af, bf, (uint32_t)tile_m, TBN);
  const uint32_t b_rows = pair ? TBN / 2 : TBN;
  const uint64_t kbg = (uint64_t)(g.K / 128);
  const uint64_t rba = (uint64_t)((g.sfa_rows + 127) / 128);
  const uint64_t rbb = (uint64_t)((g.N + 127) / 128);
  CUtensorMap ta, tb, tsa, tsb;
  const uint64_t dA[2] = {(uint64_t)g.K, (uint64_t)g.M};
  const uint64_t strideK[1] = {(uint64_t)g.K};
  const uint32_t boxA[2] = {BKB, BM};
  int rc = make_tmap(&ta, g.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dA, strideK, boxA, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  {
    const uint64_t d[3] = {128, kbg, rba};
    const uint64_t st[2] = {512, 512 * kbg};
    const uint32_t box[3] = {128, 1, 1};
    rc = make_tmap(&tsa, g.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, d, st, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  }
  if (g.mode == FP8_GROUPED_JAGGED_M) {
    const uint64_t dB[3] = {(uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.E};
    const uint64_t sB_[2] = {(uint64_t)g.K, (uint64_t)(g.N * g.K)};
    const uint32_t boxB[3] = {BKB, b_rows, 1};
    rc = make_tmap(&tb, g.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, dB, sB_, boxB, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    const uint64_t d[4] = {128, kbg, rbb, (uint64_t)g.E};
    const uint64_t st[3] = {512, 512 * kbg, 512 * kbg * rbb};
    const uint32_t box[4] = {128, 1, 2, 1};
    rc = make_tmap(&tsb, g.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, d, st, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
    p.total_rows = g.M;
    return pair ? run<kMX, kJagM, 0, 0, 2>(ta, tb, to, tsa, tsb, p, 0, c)
                : run<kMX, kJagM, 0, 0, 1>(ta, tb, to, tsa, tsb, p, 0, c);
  }
  const uint64_t dB[2] = {(uint64_t)g.K, (uint64_t)g.N};
  const uint32_t boxB[2] = {BKB, b_rows};
  rc = make_tmap(&tb, g.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dB, strideK, boxB, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  {
    const uint64_t d[3] = {128, kbg, rbb};
    const uint64_t st[2] = {512, 512 * kbg};
    const uint32_t box[3] = {128, 1, 2};
    rc = make_tmap(&tsb, g.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, d, st, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  }
  if (g.mode == -1) {
    const int64_t tiles = p.num_m * p.num_n;
    return pair ? run<kMX, kDense, 0, 0, 2>(ta, tb, to, tsa, tsb, p, tiles, c)
                : run<kMX, kDense, 0, 0, 1>(ta, tb, to, tsa, tsb, p, tiles, c);
  }
  p.total_rows = -1;
  const int64_t tiles = (int64_t)g.E * p.num_m * p.num_n;
  return pair ? run<kMX, kJagK, 0, 0, 2>(ta, tb, to, tsa, tsb, p, tiles, c)
              : run<kMX, kJagK, 0, 0, 1>(ta, tb, to, tsa, tsb, p, tiles, c);
}

}  // namespace

// Pairs (CG = 2) serve problems with enough 256-row tiles to fill the GPU; small ones run on
// single CTAs (CG = 1).
int launch_gemm(const GemmArgs& g, const Ctx& c) {
  const bool fp8 = g.a_dtype != FP8_DT_BF16;
  GemmParams p = {};
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.sA = g.sA;
  p.sB = g.sB;
  p.out = g.out;
  p.out_f32 = g.out_dtype == FP8_DT_F32;
  p.status = c.status;
  p.wait_ns = c.wait_ns;
  p.test_stall = c.test_stall;
  p.row_amax = g.row_amax;
  p.col_amax = g.col_amax;
  p.amax_whole = g.amax_whole;
  p.ends = g.ends;
  p.E = (int)g.E;
  const bool mx = g.mx != 0;
  const int tbn = mx ? Cfg<kMX, 1>::TBN : (g.blockwise ? Cfg<kBLK, 1>::TBN : BN);
  p.num_n = (g.N + tbn - 1) / tbn;
  const int esz = fp8 ? 1 : 2;
  p.nkb = (g.K * esz + BKB - 1) / BKB;
  p.ldo = g.N;
  p.vec_ok = p.out_f32 ? (p.ldo % 4 == 0) : (p.ldo % 8 == 0);
  if (g.mode != -1 && (g.E < 1 || g.E > kMaxExperts)) return FP8_ERR_UNSUPPORTED;
  // pair tiles when there are at least ~one per SM pair. Blockwise scaling runs on single CTAs:
  // its per-K-block commit / promotion / release cycle ran at half the speed across a CTA pair
  // (1050 vs 560 us on 8192 x 14336 x 4096; 600 us for the pair even with the promotion's waits
  // removed, so the pair's per-block commits, not the promotion, set that pace).
  const int64_t pair_tiles = ((g.M + 255) / 256) * p.num_n * (g.mode == FP8_GROUPED_JAGGED_K ? g.E : 1);
  const bool pair = !g.blockwise && (g.mode == FP8_GROUPED_JAGGED_M ? g.M >= 2048 : pair_tiles * 2 >= c.sm_count);
  const int tile_m = pair ? 256 : 128;
  p.num_m = (g.M + tile_m - 1) / tile_m;
  // Dense tiles walk a group of M-blocks before the next N-block (or a group of N-blocks before
  // the next M-block): the group's panels (tile rows x K) are re-read by every block of the other
  // dimension, from L2 while the group fits in ~32 MB, and every group reads all of the other
  // operand once. The orientation with fewer bytes read by that count is taken. Measured on the
  // Llama3 MLP shapes (DRAM bytes read): the forward (1 MB panels) 152 MB with 16 M-blocks per
  // group, 115 MB with all 32; the grad-input and bf16 weight-gradient GEMMs (~4 MB panels)
  // 573 / 1179 MB with 16 M-blocks, 483 / 1048 MB with 8.
  {
    auto group = [](int64_t panel, int64_t blocks) {
      int64_t gsz = panel > 0 ? kGroupBytes / panel : blocks;
      if (gsz > blocks) gsz = blocks;
      return gsz < 1 ? (int64_t)1 : gsz;  // never zero: it divides the tile index
    };
    const int64_t pa = (int64_t)tile_m * g.K * esz, pb = (int64_t)tbn * g.K * esz;  // panel bytes
    const int64_t gm = group(pa, p.num_m), gn = group(pb, p.num_n);
    const int64_t by_m = p.num_m * pa + (p.num_m + gm - 1) / gm * p.num_n * pb;  // A once, B per group
    const int64_t by_n = p.num_n * pb + (p.num_n + gn - 1) / gn * p.num_m * pa;  // B once, A per group
    p.group_m = gm;
    p.group_n = by_n < by_m ? gn : 0;
  }
  // the kernels index tiles with 32-bit arithmetic
  const int64_t max_tiles = g.mode == FP8_GROUPED_JAGGED_K ? g.E * p.num_m * p.num_n
                            : g.mode == FP8_GROUPED_JAGGED_M ? (p.num_m + g.E) * p.num_n
                                                             : p.num_m * p.num_n;
  if (max_tiles >= (int64_t)1 << 31) return FP8_ERR_UNSUPPORTED;
  // output tensor map for the pairs' TMA stores: boxes of 32 rows x 128 bytes
  CUtensorMap to, none;
  memset(&to, 0, sizeof(to));
  memset(&none, 0, sizeof(none));
  p.tma_out = 0;
  if (pair && p.vec_ok && (reinterpret_cast<uintptr_t>(g.out) & 15) == 0) {
    const CUtensorMapDataType odt = p.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle osw = CU_TENSOR_MAP_SWIZZLE_128B;
    const uint32_t bx = p.out_f32 ? 32 : 64;  // 128-byte box rows
    const uint64_t oes = p.out_f32 ? 4 : 2;
    int rc;
    if (g.mode == FP8_GROUPED_JAGGED_K) {
      const uint64_t d[3] = {(uint64_t)g.N, (uint64_t)g.M, (uint64_t)g.E};
      const uint64_t st[2] = {(uint64_t)g.N * oes, (uint64_t)(g.M * g.N) * oes};
      const uint32_t box[3] = {bx, 32, 1};
      rc = make_tmap(&to, g.out, odt, 3, d, st, box, osw);
    } else {
      const uint64_t d[2] = {(uint64_t)g.N, (uint64_t)g.M};
      const uint64_t st[1] = {(uint64_t)g.N * oes};
      const uint32_t box[2] = {bx, 32};
      rc = make_tmap(&to, g.out, odt, 2, d, st, box, osw);
    }
    if (rc) return rc;
    p.tma_out = 1;
  }

  if (mx) {
    if (g.mode != FP8_GROUPED_JAGGED_K) p.tma_out = 0;  // MX stores from registers except jagged K
    return launch_mx(g, p, to, pair, tile_m, c);
  }
  if (fp8) {
    const uint32_t af = g.a_dtype == FP8_DT_E4M3 ? kFmtE4M3 : kFmtE5M2;
    const uint32_t bf = g.b_dtype == FP8_DT_E4M3 ? kFmtE4M3 : kFmtE5M2;
    p.idesc = make_idesc(af, bf, 0, 0, tile_m, BN);
    p.sa_scalar = g.sA_len == 1;
    p.sb_scalar = g.sB_len == 1;
    CUtensorMap ta, tb;
    const uint32_t boxA[2] = {BKB, BM};
    const uint64_t dA[2] = {(uint64_t)g.K, (uint64_t)g.M};
    const uint64_t strideK[1] = {(uint64_t)g.K};
    const uint32_t b_rows = pair ? BN / 2 : BN;
    int rc = make_tmap(&ta, g.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dA, strideK, boxA, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
    if (g.mode == -1 || g.mode == FP8_GROUPED_JAGGED_K) {
      const uint64_t dB[2] = {(uint64_t)g.K, (uint64_t)g.N};
      const uint32_t boxB[2] = {BKB, b_rows};
      rc = make_tmap(&tb, g.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dB, strideK, boxB, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc) return rc;
      if (g.mode == -1) {
        const int64_t tiles = p.num_m * p.num_n;
        if (g.blockwise) {  // sA [M, K/128], sB [ceil(N/128), K/128]; 128-column tiles
          if (g.K % 128 || p.row_amax || p.col_amax) return FP8_ERR_UNSUPPORTED;
          constexpr int TB = Cfg<kBLK, 1>::TBN;
          p.idesc = make_idesc(af, bf, 0, 0, tile_m, TB);
          const uint32_t boxB2[2] = {BKB, pair ? TB / 2 : TB};
          CUtensorMap tbb;
          rc = make_tmap(&tbb, g.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dB, strideK, boxB2, CU_TENSOR_MAP_SWIZZLE_128B);
          if (rc) return rc;
          return run<kBLK, kDense, 0, 0, 1>(ta, tbb, to, none, none, p, tiles, c);
        }
        if (p.row_amax || p.col_amax)
          return pair ? run<kFP8, kDenseAmax, 0, 0, 2>(ta, tb, to, none, none, p, tiles, c)
                      : run<kFP8, kDenseAmax, 0, 0, 1>(ta, tb, to, none, none, p, tiles, c);
        if (g.q_out) {
          p.q_out = static_cast<uint8_t*>(g.q_out);
          p.q_scales = g.q_scales;
          p.q_mx = g.q_mx;
          p.q_fmt = g.q_fmt;
          p.q_tab = scale_tab(g.q_fmt);
          return pair ? run<kFP8, kDenseQuant, 0, 0, 2>(ta, tb, to, none, none, p, tiles, c)
                      : run<kFP8, kDenseQuant, 0, 0, 1>(ta, tb, to, none, none, p, tiles, c);
        }
        return pair ? run<kFP8, kDense, 0, 0, 2>(ta, tb, to, none, none, p, tiles, c) : run<kFP8, kDense, 0, 0, 1>(ta, tb, to, none, none, p, tiles, c);
      }
      if (g.blockwise) return FP8_ERR_UNSUPPORTED;
      // jagged K: A = G^T [N_out, P], B = X^T [Kd, P]; tile space M = N_out, N = Kd; the
      // offsets are checked for order and for fitting the padded length P.
      p.total_rows = -1;
      const int64_t tiles = (int64_t)g.E * p.num_m * p.num_n;
      return pair ? run<kFP8, kJagK, 0, 0, 2>(ta, tb, to, none, none, p, tiles, c) : run<kFP8, kJagK, 0, 0, 1>(ta, tb, to, none, none, p, tiles, c);
    }
    if (g.mode == FP8_GROUPED_JAGGED_M) {
      if (g.blockwise) return FP8_ERR_UNSUPPORTED;
      p.total_rows = g.M;
      const uint64_t dB[3] = {(uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.E};
      const uint64_t sB_[2] = {(uint64_t)g.K, (uint64_t)(g.N * g.K)};
      const uint32_t boxB[3] = {BKB, b_rows, 1};
      rc = make_tmap(&tb, g.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, dB, sB_, boxB, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc) return rc;
      if (!pair) return run<kFP8, kJagM, 0, 0, 1>(ta, tb, to, none, none, p, 0, c);
      // An expert's last tile with fewer than 256 rows runs transposed: the expert's 256 weight
      // rows as the MMA's M, the tile's rows rounded up to 16 as its N, and only the row boxes
      // that cover them loaded (32, 64 or 128 rows per CTA), so a short tail costs the MMAs and
      // the operand bytes of its rows, not of 256.
      CUtensorMap t32, t64;
      const uint32_t box32[2] = {BKB, 32}, box64[2] = {BKB, 64};
      rc = make_tmap(&t32, g.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dA, strideK, box32, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc) return rc;
      rc = make_tmap(&t64, g.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dA, strideK, box64, CU_TENSOR_MAP_SWIZZLE_128B);
      if (rc) return rc;
      p.tail_t = 1;
      p.idesc_t = make_idesc(bf, af, 0, 0, 256, 0);
      return run<kFP8, kJagM, 0, 0, 2>(ta, tb, to, t32, t64, p, 0, c);
    }
    return FP8_ERR_INVALID_ARG;
  }

  // BF16 (dense only)
  if (g.mode != -1) return FP8_ERR_UNSUPPORTED;
  p.idesc = make_idesc(kFmtBF16, kFmtBF16, (uint32_t)g.a_mn, (uint32_t)g.b_mn, tile_m, BN);
  const uint32_t b_rows = pair ? BN / 2 : BN;
  CUtensorMap ta, tb;
  int rc;
  if (g.a_mn) {
    const uint64_t d[2] = {(uint64_t)g.M, (uint64_t)g.K};
    const uint64_t s[1] = {(uint64_t)g.M * 2};
    const uint32_t box[2] = {64, 64};
    rc = make_tmap(&ta, g.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, s, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const uint64_t d[2] = {(uint64_t)g.K, (uint64_t)g.M};
    const uint64_t s[1] = {(uint64_t)g.K * 2};
    const uint32_t box[2] = {64, BM};
    rc = make_tmap(&ta, g.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, s, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (rc) return rc;
  if (g.b_mn) {
    const uint64_t d[2] = {(uint64_t)g.N, (uint64_t)g.K};
    const uint64_t s[1] = {(uint64_t)g.N * 2};
    const uint32_t box[2] = {64, 64};
    rc = make_tmap(&tb, g.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, s, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const uint64_t d[2] = {(uint64_t)g.K, (uint64_t)g.N};
    const uint64_t s[1] = {(uint64_t)g.K * 2};
    const uint32_t box[2] = {64, b_rows};
    rc = make_tmap(&tb, g.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, s, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (rc) return rc;
  const int64_t tiles = p.num_m * p.num_n;
  if (p.row_amax || p.col_amax) {  // side outputs: the weight-gradient layout (both MN-major) only
    if (!(g.a_mn && g.b_mn)) return FP8_ERR_UNSUPPORTED;
    return pair ? run<kBF16, kDenseAmax, 1, 1, 2>(ta, tb, to, none, none, p, tiles, c)
                : run<kBF16, kDenseAmax, 1, 1, 1>(ta, tb, to, none, none, p, tiles, c);
  }
  if (pair) {
    if (g.a_mn && g.b_mn) return run<kBF16, kDense, 1, 1, 2>(ta, tb, to, none, none, p, tiles, c);
    if (g.a_mn) return run<kBF16, kDense, 1, 0, 2>(ta, tb, to, none, none, p, tiles, c);
    if (g.b_mn) return run<kBF16, kDense, 0, 1, 2>(ta, tb, to, none, none, p, tiles, c);
    return run<kBF16, kDense, 0, 0, 2>(ta, tb, to, none, none, p, tiles, c);
  }
  if (g.a_mn && g.b_mn) return run<kBF16, kDense, 1, 1, 1>(ta, tb, to, none, none, p, tiles, c);
  if (g.a_mn) return run<kBF16, kDense, 1, 0, 1>(ta, tb, to, none, none, p, tiles, c);
  if (g.b_mn) return run<kBF16, kDense, 0, 1, 1>(ta, tb, to, none, none, p, tiles, c);
  return run<kBF16, kDense, 0, 0, 1>(ta, tb, to, none, none, p, tiles, c);
}

}  // namespace fp8lin
