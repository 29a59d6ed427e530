// Column-wise FP8 quantization (sm_103a): per column, or per column of each expert / segment,
// amax -> fp64 scale (by table) -> fp32 multiply -> clamp -> RNE saturating cast, written
// column-major ([C, rows]) for the MN-major operands of the backward GEMMs.
//
// Recipe: "FP8 Training: Quantization, Autograd, Torchao", section 2 "The quantization math".
// Layout: "FP8 training on AMD GPUs with TorchTitan and TorchAO", "Triton Kernel Optimization",
// Level 2 (column-wise scales; the output tile transposed on chip so that the column-major
// writes are coalesced) and Level 3 (relaxed atomics for the commutative amax reduction).
//
// A column's scale needs the whole column's amax before its first element can be cast, so every
// element is read twice. The two reads run at the same time, as two pipelines in each CTA of one
// persistent cooperative launch (one CTA per SM):
//   pass 1 (amax): a producer warp streams 256-row x 64-column tiles ("units") from HBM through a
//     TMA ring (128-byte swizzle; the loads keep their lines in L2); 4 warps fold each tile's
//     column maxima by shuffles and shared memory and store them as the unit's partial: 64
//     16-bit maxima, each with bit 15 set ("written"; bf16 magnitudes leave it free), in a
//     workspace the launcher zeroed;
//   pass 2 (cast): a second producer warp streams the same units again, now from L2, through its
//     own ring; three gatherer warps take each unit's strip maxima from the partials of the strip's
//     row tiles, polling (bounded) until every field reads as written, so no fence, counter or
//     barrier separates the passes; 8 warps each take 32 rows of a tile: a lane per column pair,
//     scale by table, cast in registers, write the transposed 64 x 32 box to the warp's staging
//     buffer and store it by TMA (no barrier across warps).
// Units are ordered group, chunk, row tile, strip (a chunk: whole 64-column strips of one group,
// a few MB; neighbouring CTAs read neighbouring strips of the same rows: long DRAM row segments)
// and dealt round-robin, in the same order in both passes, so a tile's second read is by the SM
// that made the first. Pass 1 may run at most a fixed number of units ahead of pass 2 (and never
// into a chunk before pass 2 has reached the chunks before it), which keeps every tile between
// its two reads in L2 whatever the tensor's size, and cannot deadlock: a chunk's pass 1 waits only
// for the pass 2 of earlier chunks, whose pass 1 is complete.
// With the maxima given (fp8_quantize_from_amax) the launch runs pass 2 alone.
#include "common.cuh"
#include "internal.h"

namespace fp8lin {

namespace {

constexpr int kCqTile = 256;                  // rows per unit (two 128-row blocks)
constexpr int kCqStageBytes = kCqTile * 128;  // 256 rows x 64 bf16
constexpr int kCqMaxStages = 4;               // per ring
constexpr int kCqP1Warps = 4;                 // pass-1 (amax) warps
constexpr int kCqP2Warps = 8;                 // pass-2 (cast) warps, 32 rows each
constexpr int kCqP1Threads = 32 * kCqP1Warps;
constexpr int kCqGathers = 3;                 // pass-2 warps gathering the maxima (unit k: warp k % gathers)
constexpr int kCqBatch = 4;                   // partials a gatherer lane loads at once (4 and 8 timed alike)
constexpr int kCqP1Warp0 = 2 + kCqGathers;    // warps: 0, 1 producers; gatherers; pass 1; pass 2
constexpr int kCqP2Warp0 = kCqP1Warp0 + kCqP1Warps;
constexpr int kCqThreads = 32 * (kCqP2Warp0 + kCqP2Warps);
constexpr uint32_t kCqWritten = 0x80008000u;  // a partial's 16-bit fields carry bit 15 once written
constexpr int kCqBox = 64 * 32;               // a pass-2 warp's staging box: 64 columns x 32 rows of codes
constexpr int kCqChunkUnits = 256;            // units per chunk: 8 MB of input
constexpr int kCqLagUnits = 1024;             // pass 1 leads pass 2 by at most 32 MB of input
constexpr int kCqMaxSegments = 2048;          // segment tables live in shared memory
constexpr uint64_t kCqDrainNs = 2000000000ull;  // fixed bound: loads in flight before exit

struct CqParams {
  const int32_t* ends;  // segment mode: end row of each segment
  int64_t C, n_groups, group_rows;
  int32_t n_strips;
  int32_t mode;         // 0: 2-D [C, R] output; 1: batched [B, C, R]; 2: segments [C, P]
  const uint32_t* amax;  // given maxima: fp32 words [n_groups, C] holding bf16 values (pass 2 alone)
  int32_t given;         // 1: the maxima are given
  uint32_t* part;        // per unit: its 64 column maxima, 32 packed words (zeroed by the launcher)
  float* inv;
  int32_t* status;
  uint64_t wait_ns;
  int32_t chunk_units, lag_units, stages_a, stages_b;
  int32_t gathers;      // gatherer warps in use: at most stages_b (see the gatherers)
  int32_t test_stall;   // failure-detection test hook: no partial ever reads as written
};

// A group of n rows: row tiles, strips per chunk and chunks (the strips split as evenly as the
// chunk size allows; all chunks but the last have sc strips).
struct CqShape {
  int32_t rt_n, sc, nch;
};
FP8_DEVI CqShape cq_shape(int64_t n, int32_t n_strips, int32_t chunk_units) {
  CqShape s;
  s.rt_n = (int32_t)((n + kCqTile - 1) / kCqTile);
  if (s.rt_n == 0) {
    s.sc = 1;
    s.nch = 0;
    return s;
  }
  int32_t sc = chunk_units / s.rt_n;
  sc = sc < 1 ? 1 : (sc > n_strips ? n_strips : sc);
  int32_t nch = (n_strips + sc - 1) / sc;
  sc = (n_strips + nch - 1) / nch;
  s.sc = sc;
  s.nch = (n_strips + sc - 1) / sc;
  return s;
}

struct CqUnit {
  int32_t g, rt, c0, valid, wrows, pstart, chunk_first, row;
  int32_t pbase, rtn;  // the unit's strip: its first partial (row tile 0) and its row tiles
};

// Segment tables in shared memory (segment mode): [0, n] unit starts, [n + 1, 2n + 1] padded
// output starts, [2n + 2, 3n + 2] first rows.
// Unit i -> group, chunk, row tile, strip. Unit and row indices fit 32 bits (the host checks).
FP8_DEVI CqUnit cq_unit(const CqParams& p, int32_t i, const int32_t* pre, const CqShape& dense) {
  int32_t g, ufirst, g0, pstart, n, wend;
  CqShape sh;
  if (p.mode == 2) {
    const int32_t ng = (int32_t)p.n_groups;
    int lo = 0, hi = ng - 1;
    while (lo < hi) {  // the last segment whose first unit is <= i (empty segments have none)
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    g = lo;
    ufirst = pre[g];
    pstart = pre[ng + 1 + g];
    g0 = pre[2 * ng + 2 + g];
    n = pre[2 * ng + 2 + g + 1] - g0;
    wend = (n + 127) & ~127;
    sh = cq_shape(n, p.n_strips, p.chunk_units);
  } else {
    sh = dense;
    const int32_t per = sh.rt_n * p.n_strips;
    g = i / per;
    ufirst = g * per;
    n = (int32_t)p.group_rows;
    g0 = g * n;
    pstart = 0;
    wend = n;
  }
  const int32_t local = i - ufirst;
  const int32_t span = sh.rt_n * sh.sc;  // units of a full chunk
  const int32_t j = local / span;        // the last, narrower chunk follows the full ones
  const int32_t rem = local - j * span;
  const int32_t w = min(sh.sc, p.n_strips - j * sh.sc);
  const int32_t rt = rem / w;
  CqUnit u;
  const int32_t strip = j * sh.sc + (rem - rt * w);
  u.g = g;
  u.rt = rt * kCqTile;
  u.c0 = strip * 64;
  u.pbase = ufirst + strip * sh.rt_n;  // a group's partials: strip-major, so a strip's are contiguous
  u.rtn = sh.rt_n;
  u.valid = min(max(n - u.rt, 0), kCqTile);
  u.wrows = min(max(wend - u.rt, 0), kCqTile);
  u.pstart = pstart;
  u.chunk_first = ufirst + j * span;
  u.row = g0 + u.rt;
  return u;
}

// Validates the offsets and builds the segment tables (segment mode); the number of units.
// False after reporting bad offsets (every thread returns the same).
FP8_DEVI bool cq_setup(const CqParams& p, int32_t* pre, const CqShape& dense, int32_t* units) {
  if (p.mode != 2) {
    *units = (int32_t)p.n_groups * dense.rt_n * p.n_strips;
    return true;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t ng = (int32_t)p.n_groups;
  int bad = 0;
  for (int32_t e = tid; e < ng; e += blockDim.x) {
    const int32_t cur = p.ends[e], prev = e ? p.ends[e - 1] : 0;
    if (cur < prev || (e == ng - 1 && (int64_t)cur != p.group_rows)) bad = 1;
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (blockIdx.x == 0 && tid == 0) set_status(p.status, FP8_DEV_BAD_OFFSETS);
    return false;
  }
  if (warp == 0) {
    int32_t cu = 0, cp = 0;
    for (int32_t base = 0; base < ng; base += 32) {
      const int32_t i = base + lane;
      int32_t vu = 0, vp = 0;
      if (i < ng) {
        const int32_t n = p.ends[i] - (i ? p.ends[i - 1] : 0);
        vu = (int32_t)((n + kCqTile - 1) / kCqTile) * p.n_strips;
        vp = (n + 127) & ~127;
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t yu = __shfl_up_sync(0xffffffffu, vu, o);
        const int32_t yp = __shfl_up_sync(0xffffffffu, vp, o);
        if (lane >= o) {
          vu += yu;
          vp += yp;
        }
      }
      if (i < ng) {
        pre[i + 1] = vu + cu;
        pre[ng + 1 + i + 1] = vp + cp;
        pre[2 * ng + 2 + i + 1] = p.ends[i];
      }
      cu += __shfl_sync(0xffffffffu, vu, 31);
      cp += __shfl_sync(0xffffffffu, vp, 31);
    }
    if (lane == 0) {
      pre[0] = 0;
      pre[ng + 1] = 0;
      pre[2 * ng + 2] = 0;
    }
  }
  __syncthreads();
  *units = pre[ng];
  return true;
}

// What a producer publishes with each stage.
struct CqInfo {
  int32_t g, c0, rt, valid, wrows, pstart, pidx;
};
struct CqShared {
  uint64_t full_a[kCqMaxStages];   // pass 1: the tile landed
  uint64_t empty_a[kCqMaxStages];  // pass 1: the amax warps are done with the stage
  uint64_t full_b[kCqMaxStages];   // pass 2: the tile landed and its maxima were gathered (2 arrivals)
  uint64_t empty_b[kCqMaxStages];  // pass 2: the cast warps are done with the stage
  CqInfo info_a[kCqMaxStages], info_b[kCqMaxStages];
  uint32_t am[kCqMaxStages][32];   // pass 2: the stage's 64 column maxima, packed bf16 pairs
  uint32_t red[kCqP1Warps][8][4];
  int32_t p2_next;                 // this CTA's next pass-2 unit: all of its units below are issued
  int abort;
};

FP8_DEVI void cq_fail(volatile int* abort, int32_t* status) {
  if (!*abort) {
    *abort = 1;
    set_status(status, FP8_DEV_TIMEOUT);
  }
}

// Bounded wait until this CTA's pass 2 has issued every unit below `target`.
FP8_DEVI bool cq_wait_lead(const volatile int32_t* p2_next, int32_t target, const volatile int* abort,
                           uint64_t limit_ns) {
  if (*p2_next >= target) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    __nanosleep(64);
    if (*p2_next >= target) return true;
    if (*abort || globaltimer() - t0 > limit_ns) return false;
  }
}

// The 16-byte vector at p (gpu scope: another SM's stores become visible to it).
FP8_DEVI uint4 ld_relaxed_v4(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
FP8_DEVI void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int FMT>
__global__ void __launch_bounds__(kCqThreads, 1) colpipe_kernel(const __grid_constant__ CUtensorMap tm_in,
                                                                const __grid_constant__ CUtensorMap tm_out,
                                                                const CqParams p,
                                                                const __grid_constant__ ScaleTab tab) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring_a = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring_b = ring_a + p.stages_a * kCqStageBytes;
  uint8_t* boxes = ring_b + p.stages_b * kCqStageBytes;
  CqShared& S = *reinterpret_cast<CqShared*>(boxes + kCqP2Warps * kCqBox);
  int32_t* pre = reinterpret_cast<int32_t*>(&S + 1);
  __shared__ ScaleTab stab;  // the lanes of a warp look up different entries at once
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const CqShape dense = p.mode == 2 ? CqShape{0, 1, 0} : cq_shape(p.group_rows, p.n_strips, p.chunk_units);
  int32_t M;
  if (!cq_setup(p, pre, dense, &M)) return;
  static_assert(sizeof(ScaleTab) % 4 == 0, "table words");
  for (int i = tid; i < (int)(sizeof(ScaleTab) / 4); i += blockDim.x)
    reinterpret_cast<uint32_t*>(&stab)[i] = reinterpret_cast<const uint32_t*>(&tab)[i];
  const int32_t cnt = (int32_t)blockIdx.x < M ? (M - 1 - (int32_t)blockIdx.x) / (int32_t)gridDim.x + 1 : 0;
  if (tid == 0) {
    for (int s = 0; s < kCqMaxStages; ++s) {
      mbar_init(&S.full_a[s], 1);
      mbar_init(&S.empty_a[s], kCqP1Warps);
      mbar_init(&S.full_b[s], 2);
      mbar_init(&S.empty_b[s], kCqP2Warps);
    }
    fence_mbar_init();
    S.abort = 0;
    S.p2_next = cnt > 0 ? (int32_t)blockIdx.x : INT32_MAX;
    tma_prefetch_desc(&tm_in);
    tma_prefetch_desc(&tm_out);
  }
  // Groups without rows have no units: their inverse scales (amax 0) are written here.
  if (blockIdx.x == 0) {
    const Scale s0 = tab_scale(tab, 0u);
    for (int64_t g = 0; g < p.n_groups; ++g) {
      const int64_t n = p.mode == 2 ? p.ends[g] - (g ? p.ends[g - 1] : 0) : p.group_rows;
      if (n > 0) continue;
      for (int64_t c = tid; c < p.C; c += blockDim.x) p.inv[g * p.C + c] = s0.inv32;
    }
  }
  __syncthreads();
  volatile int* abort = &S.abort;
  volatile int32_t* p2_next = &S.p2_next;

  if (warp == 0) {
    // ============ pass-1 producer: one lane streams the CTA's units from HBM by TMA ============
    if (lane == 0 && !p.given) {
      const uint64_t pol = l2_evict_last();  // read again by pass 2
      int s = 0;
      uint32_t ph = 0;
      int32_t k = 0;
      CqUnit nx = {};
      if (cnt > 0) nx = cq_unit(p, (int32_t)blockIdx.x, pre, dense);
      for (; k < cnt; ++k) {
        const int32_t i = (int32_t)blockIdx.x + k * (int32_t)gridDim.x;
        const CqUnit u = nx;
        if (k + 1 < cnt) nx = cq_unit(p, i + (int32_t)gridDim.x, pre, dense);
        // the lead over pass 2: at most lag units, and no unit of a chunk before pass 2 has
        // issued everything below the chunk
        const int32_t lead = min(i - p.lag_units, u.chunk_first);
        if (!cq_wait_lead(p2_next, lead, abort, p.wait_ns) || !mbar_wait(&S.empty_a[s], ph ^ 1, abort, p.wait_ns)) {
          cq_fail(abort, p.status);
          break;
        }
        S.info_a[s] = CqInfo{u.g, u.c0, u.rt, u.valid, u.wrows, u.pstart, u.pbase + u.rt / kCqTile};
        mbar_arrive_expect_tx(&S.full_a[s], kCqStageBytes);
        tma_load_2d_hint(ring_a + s * kCqStageBytes, &tm_in, &S.full_a[s], u.c0, u.row, pol);
        if (++s == p.stages_a) {
          s = 0;
          ph ^= 1;
        }
      }
      // the loads in flight land before the CTA may leave (all consumed unless aborted)
      for (int32_t j = k > p.stages_a ? k - p.stages_a : 0; j < k; ++j)
        mbar_wait(&S.full_a[j % p.stages_a], (uint32_t)((j / p.stages_a) & 1), nullptr, kCqDrainNs);
    }
  } else if (warp == 1) {
    // ============ pass-2 producer: one lane streams the CTA's units again (from L2) ============
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();  // the tile's last use
      int s = 0;
      uint32_t ph = 0;
      int32_t k = 0;
      for (; k < cnt; ++k) {
        const int32_t i = (int32_t)blockIdx.x + k * (int32_t)gridDim.x;
        const CqUnit u = cq_unit(p, i, pre, dense);
        if (!mbar_wait(&S.empty_b[s], ph ^ 1, abort, p.wait_ns)) {
          cq_fail(abort, p.status);
          break;
        }
        S.info_b[s] = CqInfo{u.g, u.c0, u.rt, u.valid, u.wrows, u.pstart, 0};
        mbar_arrive_expect_tx(&S.full_b[s], kCqStageBytes);
        tma_load_2d_hint(ring_b + s * kCqStageBytes, &tm_in, &S.full_b[s], u.c0, u.row, pol);
        *p2_next = i + (int32_t)gridDim.x;
        if (++s == p.stages_b) {
          s = 0;
          ph ^= 1;
        }
      }
      for (int32_t j = k > p.stages_b ? k - p.stages_b : 0; j < k; ++j)  // loads in flight land before exit
        mbar_wait(&S.full_b[j % p.stages_b], (uint32_t)((j / p.stages_b) & 1), nullptr, kCqDrainNs);
    }
  } else if (warp < kCqP1Warp0) {
    // = pass-2 gatherers: each unit's 64 column maxima into its stage (unit k: warp k % gathers) =
    // A strip's maxima are the maxima of its row tiles' partials, each written once by pass 1
    // with bit 15 set in every 16-bit field: a field without it is not written yet, so the warp
    // polls (bounded) until all are, with no counter or fence between the passes. Lane l reads
    // 16-byte vector l % 8 (8 columns) of the row tiles l / 8, l / 8 + 4, ...
    // The gatherers wait on the stages' empty barriers out of order; a parity wait is exact only
    // while its waiter is at most one phase ahead, which holds when gathers <= stages_b: a warp's
    // previous unit k - gathers needed unit k - gathers - stages_b consumed, and the cast warps
    // consume in order, so the stage's use before the previous one is complete.
    const int gw = warp - 2;
    const int q = lane & 7, r0 = lane >> 3;
    for (int32_t k = gw; k < cnt && gw < p.gathers; k += p.gathers) {
      const int s = k % p.stages_b;
      const CqUnit u = cq_unit(p, (int32_t)blockIdx.x + k * (int32_t)gridDim.x, pre, dense);
      const bool free = lane == 0 ? mbar_wait(&S.empty_b[s], (uint32_t)(((k / p.stages_b) & 1) ^ 1), abort, p.wait_ns) : true;
      if (!__shfl_sync(0xffffffffu, free, 0)) {
        if (lane == 0) cq_fail(abort, p.status);
        break;
      }
      if (p.given) {  // the caller's fp32 words hold bf16 values: their upper halves
        const uint32_t* arow = p.amax + (int64_t)u.g * p.C;
        const int64_t col = u.c0 + 2 * lane;
        const uint32_t lo = col < p.C ? arow[col] >> 16 : 0u, hi = col + 1 < p.C ? arow[col + 1] >> 16 : 0u;
        S.am[s][lane] = (lo & 0x7FFFu) | ((hi & 0x7FFFu) << 16);
      } else {
        const uint32_t* base = p.part + (int64_t)u.pbase * 32 + 4 * q;
        uint4 acc = make_uint4(0, 0, 0, 0);
        bool ok = true;
        // kCqBatch partials per lane in flight at once (a tall strip has one per row tile; rows
        // past the strip count as written zeros). A batch that is not all written yet is taken
        // again entry by entry, each polled (bounded) until written.
        for (int32_t r = r0; r < u.rtn && ok; r += 4 * kCqBatch) {
          uint4 v[kCqBatch];
#pragma unroll
          for (int j = 0; j < kCqBatch; ++j)
            v[j] = r + 4 * j < u.rtn ? ld_relaxed_v4(base + (int64_t)(r + 4 * j) * 32)
                                     : make_uint4(kCqWritten, kCqWritten, kCqWritten, kCqWritten);
          uint32_t all = p.test_stall ? 0u : kCqWritten;
#pragma unroll
          for (int j = 0; j < kCqBatch; ++j) all &= v[j].x & v[j].y & v[j].z & v[j].w;
          if (all == kCqWritten) {
#pragma unroll
            for (int j = 0; j < kCqBatch; ++j)
              acc = make_uint4(__vmaxu2(acc.x, v[j].x), __vmaxu2(acc.y, v[j].y), __vmaxu2(acc.z, v[j].z),
                               __vmaxu2(acc.w, v[j].w));
            continue;
          }
#pragma unroll 1
          for (int32_t rr = r; rr < u.rtn && rr < r + 4 * kCqBatch && ok; rr += 4) {
            uint4 w = ld_relaxed_v4(base + (int64_t)rr * 32);
            bool done = !p.test_stall && ((w.x & w.y & w.z & w.w & kCqWritten) == kCqWritten);
            if (!done) {
              const uint64_t t0 = globaltimer();
              while (!done) {
                __nanosleep(64);
                w = ld_relaxed_v4(base + (int64_t)rr * 32);
                done = !p.test_stall && ((w.x & w.y & w.z & w.w & kCqWritten) == kCqWritten);
                if (!done && (*abort || globaltimer() - t0 > p.wait_ns)) {
                  ok = false;
                  break;
                }
              }
            }
            acc = make_uint4(__vmaxu2(acc.x, w.x), __vmaxu2(acc.y, w.y), __vmaxu2(acc.z, w.z), __vmaxu2(acc.w, w.w));
          }
        }
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) cq_fail(abort, p.status);
          break;
        }
#pragma unroll
        for (int d = 8; d <= 16; d <<= 1) {
          acc.x = __vmaxu2(acc.x, __shfl_xor_sync(0xffffffffu, acc.x, d));
          acc.y = __vmaxu2(acc.y, __shfl_xor_sync(0xffffffffu, acc.y, d));
          acc.z = __vmaxu2(acc.z, __shfl_xor_sync(0xffffffffu, acc.z, d));
          acc.w = __vmaxu2(acc.w, __shfl_xor_sync(0xffffffffu, acc.w, d));
        }
        if (lane < 8)
          *reinterpret_cast<uint4*>(&S.am[s][4 * q]) = make_uint4(acc.x & 0x7FFF7FFFu, acc.y & 0x7FFF7FFFu,
                                                                  acc.z & 0x7FFF7FFFu, acc.w & 0x7FFF7FFFu);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.full_b[s]);
    }
  } else if (warp < kCqP2Warp0) {
    // ============ pass-1 amax warps: thread = 4 rows x 8 columns of 4 row groups per tile ============
    if (!p.given) {
      const int ct = tid - 32 * kCqP1Warp0, cw = ct >> 5;
      const int ch = lane & 7, rq = lane >> 3;
      int s = 0;
      uint32_t ph = 0;
      for (int32_t k = 0; k < cnt; ++k) {
        const bool got = mbar_wait(&S.full_a[s], ph, abort, p.wait_ns);
        if (!named_bar_and(2, kCqP1Threads, got)) {  // uniform decision across the amax warps
          if (!got) cq_fail(abort, p.status);
          break;
        }
        const CqInfo info = S.info_a[s];
        const uint8_t* st = ring_a + s * kCqStageBytes;
        uint4 v[16];  // b: 128-row block b / 8, then 16-row half, then row of 4
        if (info.valid == kCqTile) {
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            const int r = 128 * (b >> 3) + 32 * cw + 16 * ((b >> 2) & 1) + 4 * rq + (b & 3);
            v[b] = *reinterpret_cast<const uint4*>(st + r * 128 + ((ch ^ (r & 7)) << 4));
          }
        } else {
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            const int r = 128 * (b >> 3) + 32 * cw + 16 * ((b >> 2) & 1) + 4 * rq + (b & 3);
            v[b] = r < info.valid ? *reinterpret_cast<const uint4*>(st + r * 128 + ((ch ^ (r & 7)) << 4))
                                  : make_uint4(0, 0, 0, 0);  // rows past the group read as zeros
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty_a[s]);  // this warp is done with the stage
        if (++s == p.stages_a) {
          s = 0;
          ph ^= 1;
        }
        uint32_t m4[4] = {0, 0, 0, 0};
#pragma unroll
        for (int b = 0; b < 16; ++b) {
          m4[0] = absmax2(m4[0], v[b].x);
          m4[1] = absmax2(m4[1], v[b].y);
          m4[2] = absmax2(m4[2], v[b].z);
          m4[3] = absmax2(m4[3], v[b].w);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          m4[q] = __vmaxu2(m4[q], __shfl_xor_sync(0xffffffffu, m4[q], 8));
          m4[q] = __vmaxu2(m4[q], __shfl_xor_sync(0xffffffffu, m4[q], 16));
        }
        if (rq == 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q) S.red[cw][ch][q] = m4[q];
        }
        named_bar_sync(1, kCqP1Threads);
        if (cw == 0) {  // pair t = columns 2t, 2t+1 = chunk t/4, word t%4: the unit's partial
          uint32_t m = 0;
#pragma unroll
          for (int w = 0; w < kCqP1Warps; ++w) m = __vmaxu2(m, S.red[w][lane >> 2][lane & 3]);
          st_relaxed_u32(p.part + (int64_t)info.pidx * 32 + lane, m | kCqWritten);
        }
        named_bar_sync(1, kCqP1Threads);  // red[] is free again
      }
    }
  } else {
    // ====== pass-2 cast warps: each casts 32 rows x 64 columns of a tile and stores them ======
    // Lane l owns the column pair (2 l, 2 l + 1); a 32-bit shared load holds the pair's values of
    // one row (the 128-byte swizzle permutes 16-byte chunks inside a row, so the 32 lanes still
    // read one row's 128 bytes). Its 2 x 32 codes go to the warp's staging box [64 columns][32
    // rows] and the warp's elected lane stores the box by TMA.
    const int cw = warp - kCqP2Warp0;
    const int r0 = 32 * cw;  // the warp's rows within the unit
    const uint64_t out_pol = l2_evict_first();  // the codes are not re-read here
    const uint32_t woff = ((uint32_t)(lane & 3) << 2);
    uint8_t* box = boxes + cw * kCqBox;
    int s = 0;
    uint32_t ph = 0;
    for (int32_t k = 0; k < cnt; ++k) {
      const bool got = mbar_wait(&S.full_b[s], ph, abort, p.wait_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) cq_fail(abort, p.status);
        break;
      }
      const CqInfo info = S.info_b[s];
      // the scale step for the lane's two columns (table in shared memory); the first row tile
      // of a strip also writes their inverse scales
      const uint32_t am2 = S.am[s][lane];
      const Scale sv_lo = tab_scale(stab, am2 & 0xFFFFu), sv_hi = tab_scale(stab, am2 >> 16);
      if (info.rt == 0 && cw == 0) {
        const int64_t col = info.c0 + 2 * lane;
        if (col < p.C) p.inv[(int64_t)info.g * p.C + col] = sv_lo.inv32;
        if (col + 1 < p.C) p.inv[(int64_t)info.g * p.C + col + 1] = sv_hi.inv32;
      }
      const uint8_t* st = ring_b + s * kCqStageBytes + r0 * 128 + woff;
      uint32_t w[32];
      if (info.valid >= r0 + 32) {
#pragma unroll
        for (int r = 0; r < 32; ++r)
          w[r] = *reinterpret_cast<const uint32_t*>(st + r * 128 + ((((uint32_t)lane >> 2) ^ (uint32_t)(r & 7)) << 4));
      } else {
#pragma unroll
        for (int r = 0; r < 32; ++r)  // rows past the group read as zeros
          w[r] = r0 + r < info.valid
                     ? *reinterpret_cast<const uint32_t*>(st + r * 128 + ((((uint32_t)lane >> 2) ^ (uint32_t)(r & 7)) << 4))
                     : 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty_b[s]);  // this warp is done with the stage
      if (++s == p.stages_b) {
        s = 0;
        ph ^= 1;
      }
      if (r0 >= info.wrows) continue;  // nothing of this warp's rows is written
      uint32_t olo[8], ohi[8];
      const float2 slo = make_float2(sv_lo.s32, sv_lo.s32), shi = make_float2(sv_hi.s32, sv_hi.s32);
#pragma unroll
      for (int r = 0; r < 32; r += 4) {
        // column 2 l: the low halves of rows r .. r + 3; column 2 l + 1: the high halves
        const float2 l01 = fmul2_rn(make_float2(__uint_as_float(w[r] << 16), __uint_as_float(w[r + 1] << 16)), slo);
        const float2 l23 = fmul2_rn(make_float2(__uint_as_float(w[r + 2] << 16), __uint_as_float(w[r + 3] << 16)), slo);
        const float2 h01 = fmul2_rn(make_float2(__uint_as_float(w[r] & 0xFFFF0000u), __uint_as_float(w[r + 1] & 0xFFFF0000u)), shi);
        const float2 h23 = fmul2_rn(make_float2(__uint_as_float(w[r + 2] & 0xFFFF0000u), __uint_as_float(w[r + 3] & 0xFFFF0000u)), shi);
        olo[r / 4] = cvt_fp8x2<FMT>(l01.x, l01.y) | (cvt_fp8x2<FMT>(l23.x, l23.y) << 16);
        ohi[r / 4] = cvt_fp8x2<FMT>(h01.x, h01.y) | (cvt_fp8x2<FMT>(h23.x, h23.y) << 16);
      }
      if (lane == 0) bulk_wait_read_all();  // the previous store has read the box
      __syncwarp();
      uint8_t* dst = box + lane * 64;  // rows 2 l and 2 l + 1 of the box: 32 codes each
      *reinterpret_cast<uint4*>(dst) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
      *reinterpret_cast<uint4*>(dst + 16) = make_uint4(olo[4], olo[5], olo[6], olo[7]);
      *reinterpret_cast<uint4*>(dst + 32) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
      *reinterpret_cast<uint4*>(dst + 48) = make_uint4(ohi[4], ohi[5], ohi[6], ohi[7]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int32_t xo = info.pstart + info.rt + r0;
        if (p.mode == 1)
          tma_store_3d_hint(&tm_out, box, xo, info.c0, info.g, out_pol);
        else
          tma_store_2d_hint(&tm_out, box, xo, info.c0, out_pol);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_all();
  }
  __syncthreads();
}

constexpr int kCqSmemMax = 232448;  // the opt-in shared memory of a CTA (227 KB)

size_t cq_smem(int sa, int sb, size_t pre) {
  return 1024 + (size_t)(sa + sb) * kCqStageBytes + kCqP2Warps * kCqBox + sizeof(CqShared) + pre + sizeof(ScaleTab);
}

}  // namespace

// Workspace words of a column quantize: one partial (32 words: the 64 column maxima of a
// 256-row x 64-column unit) per unit; a group of n rows has ceil(n / 256) units per 64-column
// strip, so rows_total / 256 + groups bounds the row tiles of all groups.
int64_t col_ws_words(int64_t groups, int64_t C, int64_t rows_total) {
  return (ceil_div64(rows_total, kCqTile) + groups) * ceil_div64(C, 64) * 32;
}

int launch_quant_cols(const void* x, int64_t rows_total, int64_t C, int64_t n_groups, int64_t group_rows,
                      const int32_t* ends, int fmt, void* out_t, int64_t ld_out, float* inv, uint32_t* scratch,
                      const Ctx& c, const uint32_t* amax_given) {
  if (n_groups == 0 || C == 0) return FP8_OK;
  if (ends && n_groups > kCqMaxSegments) return FP8_ERR_UNSUPPORTED;
  if (rows_total > INT32_MAX) return FP8_ERR_UNSUPPORTED;  // rows are TMA coordinates
  CqParams p = {};
  p.ends = ends;
  p.C = C;
  p.n_groups = n_groups;
  p.group_rows = ends ? rows_total : group_rows;  // segment mode: the last end must equal it
  p.n_strips = (int32_t)ceil_div64(C, 64);
  p.mode = ends ? 2 : (n_groups > 1 ? 1 : 0);
  p.inv = inv;
  p.status = c.status;
  p.wait_ns = c.wait_ns;
  p.chunk_units = kCqChunkUnits;
  p.lag_units = kCqLagUnits;
  p.test_stall = c.test_stall;

  CUtensorMap tout, tin;
  int rc;
  if (p.mode == 1) {
    const uint64_t dims[3] = {(uint64_t)group_rows, (uint64_t)C, (uint64_t)n_groups};
    const uint64_t strides[2] = {(uint64_t)group_rows, (uint64_t)(C * group_rows)};
    const uint32_t box[3] = {32, 64, 1};  // one warp's box: 32 rows (bytes) x 64 columns
    rc = make_tmap(&tout, out_t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    const uint64_t inner = p.mode == 2 ? (uint64_t)ld_out : (uint64_t)group_rows;
    const uint64_t dims[2] = {inner, (uint64_t)C};
    const uint64_t strides[1] = {(uint64_t)ld_out};
    const uint32_t box[2] = {32, 64};  // one warp's box: 32 rows (bytes) x 64 columns
    rc = make_tmap(&tout, out_t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (rc != FP8_OK) return rc;
  {
    const uint64_t dims[2] = {(uint64_t)C, (uint64_t)(rows_total > 0 ? rows_total : 1)};
    const uint64_t strides[1] = {(uint64_t)C * 2};
    const uint32_t box[2] = {64, kCqTile};
    rc = make_tmap(&tin, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != FP8_OK) return rc;
  }

  if (amax_given) {
    p.amax = amax_given;  // read only (pass 2 alone)
    p.given = 1;
  } else {  // every partial starts unwritten
    if (cudaMemsetAsync(scratch, 0, (size_t)col_ws_words(n_groups, C, rows_total) * 4, c.stream) != cudaSuccess)
      return FP8_ERR_CUDA;
    p.part = scratch;
  }
  // units: exact for dense groups; for segments an upper bound (each segment adds at most one
  // partial tile) -- the kernel computes the exact count from the offsets
  const int64_t units = ends ? (ceil_div64(rows_total, kCqTile) + n_groups) * p.n_strips
                             : n_groups * ceil_div64(group_rows, kCqTile) * p.n_strips;
  if (units > INT32_MAX - 2 * (int64_t)c.sm_count - kCqLagUnits) return FP8_ERR_UNSUPPORTED;  // 32-bit unit indices
  const size_t pre = ends ? 12 * (size_t)(n_groups + 1) : 0;
  // two rings of 32 KB stages: 3 + 3 where the segment tables leave room, else fewer
  int sa = 3, sb = 3;
  if (cq_smem(sa, sb, pre) > kCqSmemMax) sb = 2;
  if (cq_smem(sa, sb, pre) > kCqSmemMax) sa = 2;
  if (cq_smem(sa, sb, pre) > kCqSmemMax) return FP8_ERR_UNSUPPORTED;
  p.stages_a = sa;
  p.stages_b = sb;
  p.gathers = kCqGathers < sb ? kCqGathers : sb;
  const size_t smem = cq_smem(sa, sb, pre) - sizeof(ScaleTab);  // the table is static shared memory
  const int64_t grid = units > 0 ? (units < c.sm_count ? units : c.sm_count) : 1;
  const ScaleTab& tab = scale_tab(fmt);
  auto kern = fmt == FP8_DT_E4M3 ? colpipe_kernel<FP8_DT_E4M3> : colpipe_kernel<FP8_DT_E5M2>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return FP8_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: they wait on one another's maxima
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kCqThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tin, tout, p, tab) != cudaSuccess) return FP8_ERR_CUDA;
  return FP8_OK;
}

}  // namespace fp8lin
