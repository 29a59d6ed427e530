// MXFP8 block quantization on sm_103a: blocks of 32 consecutive elements along the contraction
// dimension, one E8M0 (power-of-two) scale per block.
//
// The pages name MXFP8 as the granularity that packs a scale per group with the data ("FP8
// training on AMD GPUs with TorchTitan and TorchAO", section "AMD FP8 format in TorchAO") and as
// the next step for the quantization and grouped-GEMM kernels ("Summary and Next Steps"). The
// block size, the E8M0 scale and its rule follow the OCP Microscaling Formats (MX) specification
// v1.0: X = 2^(floor(log2(amax)) - emax_elem), emax_elem = 8 (e4m3) or 15 (e5m2), the exponent
// clamped below at -127; each element is x / X, rounded to nearest even and saturated.
//
// The row-major output alone runs on row teams (mx_rows_kernel). The column-major output (blocks
// down a column, written transposed), alone or with the row-major one (blocks along a row) from a
// single read, runs on a persistent pipelined kernel over tiles of 128 rows x 128 columns
// (mx_pipe_kernel, below).
// The E8M0 scales are written in the tensor-core scale-factor layout the MX GEMM reads: for an
// operand with rows r (its non-contraction index) and K blocks j, 512-byte blocks
// [r / 128][j / 4], and inside one the code of (r, j) at byte (r % 32) * 16 + (r / 32 % 4) * 4 +
// j % 4. A tile row's four block codes therefore form one aligned 32-bit word.
// With segment offsets (MoE), tiles walk the segment-padded row space: segment e occupies padded
// rows [pstart_e, pstart_e + roundup(count_e, 128)), so blocks never straddle two segments and
// the padding quantizes as zeros.
#include "common.cuh"
#include "internal.h"

namespace fp8lin {

namespace {

constexpr int kTile = 128;             // rows and columns of a tile
constexpr int kMaxSegments = 2048;

struct MxArgs {
  const uint16_t* x;
  int64_t R, C;           // rows and columns of one batch entry (C % 128 == 0)
  uint8_t* q;             // row-major codes in x's shape, or null
  uint8_t* sf;            // their scales: [batch][rb_q][C / 128][512 B]
  int64_t rb_q;           // 128-row blocks of sf per batch entry
  uint8_t* qt;            // column-major codes [batch][C][ld_t], or null
  int64_t ld_t;           // row length of qt: R, or the padded row count P with segments
  uint8_t* sft;           // their scales: [batch][C / 128][ld_t / 128][512 B]
  const int32_t* pstart;  // segments: padded starts [E + 1] (pstart[E] = padded rows in use)
  const int32_t* ends;
  int E;
};

// Tiles of 128 x 128 bf16 through a persistent pipeline (column-major output, with or without the
// row-major one; dense, batched or segments): one CTA per SM walks its tiles (t = CTA, CTA + grid, ...; tile columns fastest,
// so neighbouring CTAs read neighbouring 256-byte pieces of the same rows); a producer warp
// streams each 128 x 128 tile into a 4-stage ring as two 128-byte-swizzled TMA boxes of 64
// columns, and 8 warps per tile
//   - row blocks: a thread per (row, block) pair twice over, four 16-byte shared loads hold the
//     block's 32 elements; four consecutive lanes hold a row's four blocks (shuffles gather the
//     scale word); the codes go straight to global memory, 32 bytes a thread;
//   - column blocks: a thread per (column pair, 32-row quarter), 32 four-byte shared loads (a
//     warp reads one 128-byte box row at a time: conflict-free); the codes go to the
//     column-major output, 32 bytes per column;
// then release the stage. Loads of the next tiles are in flight while a tile is cast (a kernel
// with one tile per CTA and no overlap inside a CTA timed 14-26% slower on dense tensors).
constexpr int kMpStages = 4;
constexpr int kMpWarps = 8;                           // consumer warps
constexpr int kMpThreads = 32 * (kMpWarps + 1);       // + the producer warp
constexpr int kMpBoxBytes = kTile * 128;              // 128 rows x 64 bf16
constexpr int kMpStageBytes = 2 * kMpBoxBytes;
constexpr uint64_t kMpDrainNs = 2000000000ull;        // fixed bound: loads in flight before exit
struct MpShared {
  uint64_t full[kMpStages];
  uint64_t empty[kMpStages];
  int abort;
};
constexpr int kMpSmem = 1024 + kMpStages * kMpStageBytes + (int)sizeof(MpShared);

struct MpTile {
  int64_t row0;   // first source row (flat over the batch entries)
  int64_t prow0;  // its row within its batch entry (scale and column-major row space)
  int64_t b, c0;
  int valid;      // source rows of the tile (rows of the next batch entry or past the tensor: masked)
};

FP8_DEVI MpTile mp_tile(const MxArgs& a, int64_t t, int64_t ncols, int64_t grid_y) {
  MpTile T;
  const int64_t tx = t % ncols, rest = t / ncols;
  const int64_t ty = rest % grid_y;
  T.b = rest / grid_y;
  T.c0 = tx * kTile;
  T.prow0 = ty * kTile;
  T.row0 = T.b * a.R + T.prow0;
  T.valid = (int)(a.R - T.prow0 < kTile ? a.R - T.prow0 : kTile);
  return T;
}

// Segments: a CTA's tiles are described once, before its loops (a thread per tile), so that no
// segment lookup sits on the producer's or the consumers' path: tile t of the padded rows in use
// (t mod ncols: its 128-column tile) finds its segment by binary search on the padded starts.
constexpr int kMpMaxTiles = 512;  // descriptors per CTA (the launcher sizes the grid to fit)
struct MpDesc {
  int32_t row0, prow0, c0, valid;
};
FP8_DEVI MpDesc mp_desc(const MxArgs& a, int64_t t, int64_t ncols) {
  MpDesc D;
  const int64_t ty = t / ncols;
  D.c0 = (int32_t)((t - ty * ncols) * kTile);
  D.prow0 = (int32_t)(ty * kTile);
  int lo = 0, hi = a.E - 1;  // the last segment whose padded start is <= prow0
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.pstart + mid) <= D.prow0) lo = mid;
    else hi = mid - 1;
  }
  const int32_t start = lo ? __ldg(a.ends + lo - 1) : 0, cnt = __ldg(a.ends + lo) - start;
  const int32_t off = D.prow0 - __ldg(a.pstart + lo);
  D.row0 = start + off;
  D.valid = cnt - off < kTile ? cnt - off : kTile;
  return D;
}

template <int FMT, bool ROWS, bool COLS, bool JAG>
__global__ void __launch_bounds__(kMpThreads, 1)
    mx_pipe_kernel(const __grid_constant__ CUtensorMap tm_x, const MxArgs a, int64_t ncols, int64_t grid_y,
                   int64_t n_tiles, int32_t* status, uint64_t wait_ns, int test_stall) {
  extern __shared__ uint8_t mp_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mp_raw) + 1023) & ~uintptr_t(1023));
  MpShared& S = *reinterpret_cast<MpShared*>(ring + kMpStages * kMpStageBytes);
  MpDesc* desc = reinterpret_cast<MpDesc*>(&S + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // segments: only the row tiles of the padded rows in use (none when the offsets were rejected)
  const int64_t n_run = JAG ? ncols * (__ldg(a.pstart + a.E) / kTile) : n_tiles;
  const int64_t cnt = (int64_t)blockIdx.x < n_run ? (n_run - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (JAG)
    for (int64_t k = tid; k < cnt; k += blockDim.x) desc[k] = mp_desc(a, blockIdx.x + k * (int64_t)gridDim.x, ncols);
  // tile k of this CTA
  auto tile_k = [&](int64_t k) {
    if (!JAG) return mp_tile(a, blockIdx.x + k * (int64_t)gridDim.x, ncols, grid_y);
    const MpDesc D = desc[k];
    MpTile T;
    T.row0 = D.row0;
    T.prow0 = D.prow0;
    T.b = 0;
    T.c0 = D.c0;
    T.valid = D.valid;
    return T;
  };
  if (tid == 0) {
    for (int s = 0; s < kMpStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kMpWarps);
    }
    fence_mbar_init();
    S.abort = 0;
    tma_prefetch_desc(&tm_x);
  }
  __syncthreads();
  volatile int* abort = &S.abort;
  auto fail = [&]() {
    if (!*abort) {
      *abort = 1;
      set_status(status, FP8_DEV_TIMEOUT);
    }
  };

  if (warp == kMpWarps) {
    // ================= producer: one lane streams the CTA's tiles by TMA =================
    // (the failure-detection test hook: no tile is loaded, so the consumers' first wait runs out)
    if (lane == 0 && !test_stall) {
      int s = 0;
      uint32_t ph = 0;
      int64_t issued = 0;
      for (int64_t k = 0; k < cnt; ++k) {
        const MpTile T = tile_k(k);
        if (!mbar_wait(&S.empty[s], ph ^ 1, abort, wait_ns)) {
          fail();
          break;
        }
        uint8_t* st = ring + s * kMpStageBytes;
        mbar_arrive_expect_tx(&S.full[s], kMpStageBytes);
        tma_load_2d(st, &tm_x, &S.full[s], (int32_t)T.c0, (int32_t)T.row0);
        tma_load_2d(st + kMpBoxBytes, &tm_x, &S.full[s], (int32_t)(T.c0 + 64), (int32_t)T.row0);
        ++issued;
        if (++s == kMpStages) {
          s = 0;
          ph ^= 1;
        }
      }
      for (int64_t i = issued > kMpStages ? issued - kMpStages : 0; i < issued; ++i)  // loads in flight land
        mbar_wait(&S.full[i % kMpStages], (uint32_t)((i / kMpStages) & 1), nullptr, kMpDrainNs);
    }
    return;
  }

  // ======================= consumers: 8 warps cast each tile =======================
  const int64_t ncb = a.C / kTile;
  int s = 0;
  uint32_t ph = 0;
  for (int64_t k = 0; k < cnt; ++k) {
    const MpTile T = tile_k(k);
    if (!__all_sync(0xffffffffu, mbar_wait(&S.full[s], ph, abort, wait_ns))) {
      if (lane == 0) fail();
      break;
    }
    const uint8_t* st = ring + s * kMpStageBytes;
    if (ROWS) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int idx = tid + 256 * h, r = idx >> 2, j = idx & 3;  // row r, block j (columns 32 j ..)
        const uint8_t* rowp = st + (j >> 1) * kMpBoxBytes + r * 128;
        const int cb = (j & 1) * 4;
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          v[i] = r < T.valid ? *reinterpret_cast<const uint4*>(rowp + (((cb + i) ^ (r & 7)) << 4))
                             : make_uint4(0, 0, 0, 0);
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) m = absmax_vec8(m, v[i]);
        const uint32_t code = mx_code<FMT>(absmax_fold(m));
        const float inv = mx_inv(code);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[2 * i] = mx_cast2<FMT>(v[i].x, inv) | (mx_cast2<FMT>(v[i].y, inv) << 16);
          o[2 * i + 1] = mx_cast2<FMT>(v[i].z, inv) | (mx_cast2<FMT>(v[i].w, inv) << 16);
        }
        const int l0 = lane & ~3;  // the row's four blocks: lanes l0 .. l0 + 3
        const uint32_t word = __shfl_sync(0xffffffffu, code, l0) | (__shfl_sync(0xffffffffu, code, l0 + 1) << 8) |
                              (__shfl_sync(0xffffffffu, code, l0 + 2) << 16) |
                              (__shfl_sync(0xffffffffu, code, l0 + 3) << 24);
        if (r < T.valid) {
          uint4* dq = reinterpret_cast<uint4*>(a.q + (T.row0 + r) * a.C + T.c0 + 32 * j);
          dq[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dq[1] = make_uint4(o[4], o[5], o[6], o[7]);
          if (j == 0) {
            const int64_t pr = T.prow0 + r;
            uint8_t* blk = a.sf + ((T.b * a.rb_q + (pr >> 7)) * ncb + (T.c0 >> 7)) * 512;
            *reinterpret_cast<uint32_t*>(blk + (pr & 31) * 16 + ((pr >> 5) & 3) * 4) = word;
          }
        }
      }
    }
    if (COLS) {
      // thread: columns 2 cp, 2 cp + 1 of the tile, rows 32 qb .. 32 qb + 31 (one block each)
      const int cp = tid & 63, qb = tid >> 6, r0 = 32 * qb;
      const uint8_t* colp = st + (cp >> 5) * kMpBoxBytes + (cp & 3) * 4;
      const int chunk = (cp & 31) >> 2;
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = r0 + i;
        w[i] = r < T.valid ? *reinterpret_cast<const uint32_t*>(colp + r * 128 + ((chunk ^ (r & 7)) << 4)) : 0u;
      }
      uint32_t m2 = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) m2 = absmax2(m2, w[i]);
      const uint32_t code_lo = mx_code<FMT>(m2 & 0xFFFFu), code_hi = mx_code<FMT>(m2 >> 16);
      const float inv_lo = mx_inv(code_lo), inv_hi = mx_inv(code_hi);
      uint32_t olo[8], ohi[8];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        // column 2 cp: the low halves of rows i .. i + 3; column 2 cp + 1: the high halves
        const uint32_t l01 = (w[i] & 0xFFFFu) | (w[i + 1] << 16), l23 = (w[i + 2] & 0xFFFFu) | (w[i + 3] << 16);
        const uint32_t h01 = (w[i] >> 16) | (w[i + 1] & 0xFFFF0000u), h23 = (w[i + 2] >> 16) | (w[i + 3] & 0xFFFF0000u);
        olo[i / 4] = mx_cast2<FMT>(l01, inv_lo) | (mx_cast2<FMT>(l23, inv_lo) << 16);
        ohi[i / 4] = mx_cast2<FMT>(h01, inv_hi) | (mx_cast2<FMT>(h23, inv_hi) << 16);
      }
      const int c = 2 * cp;
      uint4* dlo = reinterpret_cast<uint4*>(a.qt + (T.b * a.C + T.c0 + c) * a.ld_t + T.prow0 + r0);
      uint4* dhi = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(dlo) + a.ld_t);
      dlo[0] = make_uint4(olo[0], olo[1], olo[2], olo[3]);
      dlo[1] = make_uint4(olo[4], olo[5], olo[6], olo[7]);
      dhi[0] = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
      dhi[1] = make_uint4(ohi[4], ohi[5], ohi[6], ohi[7]);
      const int64_t nrb = a.ld_t / kTile;
      uint8_t* blk = a.sft + ((T.b * (a.C / kTile) + (T.c0 >> 7)) * nrb + (T.prow0 >> 7)) * 512;
      blk[(c & 31) * 16 + (c >> 5) * 4 + qb] = (uint8_t)code_lo;
      blk[((c + 1) & 31) * 16 + ((c + 1) >> 5) * 4 + qb] = (uint8_t)code_hi;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);  // this warp is done with the stage
    if (++s == kMpStages) {
      s = 0;
      ph ^= 1;
    }
  }
}

// Segment check and padded starts: pstart[e + 1] = pstart[e] + roundup(count_e, 128). Bad
// offsets (decreasing, last != rows) or a padded total above P set FP8_DEV_BAD_OFFSETS and leave
// pstart[E] = 0, so that the quantize kernel writes nothing.
__global__ void __launch_bounds__(1024) mx_pstart_kernel(const int32_t* ends, int E, int64_t rows, int64_t P,
                                                          int32_t* pstart, int32_t* status) {
  __shared__ int32_t part[32];
  __shared__ int bad_any;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) bad_any = 0;
  __syncthreads();
  // each thread owns segments 2 tid and 2 tid + 1
  int32_t pad[2];
  int bad = 0;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int e = 2 * tid + j;
    pad[j] = 0;
    if (e < E) {
      const int32_t cur = ends[e], prev = e ? ends[e - 1] : 0;
      if (cur < prev || (e == E - 1 && cur != rows)) bad = 1;
      const int32_t cnt = cur > prev ? cur - prev : 0;
      pad[j] = (cnt + 127) / 128 * 128;
    }
  }
  if (bad) atomicOr(&bad_any, 1);
  int32_t s = pad[0] + pad[1];
  int32_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) part[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = part[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    part[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int32_t excl = incl - s + (warp ? part[warp - 1] : 0);
  const int32_t total = part[31];
  const bool ok = !bad_any && total <= P;
  if (2 * tid < E) pstart[2 * tid] = excl;
  if (2 * tid + 1 < E) pstart[2 * tid + 1] = excl + pad[0];
  if (tid == 0) {
    pstart[E] = ok ? total : 0;
    if (!ok) set_status(status, FP8_DEV_BAD_OFFSETS);
  }
}

// Row-major output alone: teams of WPR warps per row walk the rows (grid-stride), like the
// row-wise FP8 kernel: a lane holds vectors t, t + TPR, ... of 8 bf16, so the four lanes 4k .. 4k + 3
// of a load step hold one block of 32 (two shuffles give its amax) and 16 lanes hold one
// 128-column scale word (four block codes gathered by shuffles, written by the first lane).
// With segments the scales go to the padded row of the row's segment (pstart[e] + row - start_e);
// the team's rows increase, so its segment index only moves forward.
constexpr int kMxRowVPL = 16;  // vectors of 8 per lane: rows of up to 16 * 32 * WPR * 8 elements
template <int FMT, int WPR, bool JAG>
__global__ void __launch_bounds__(256) mx_rows_kernel(const uint4* __restrict__ x, int64_t rows, int64_t R,
                                                      int nvec, uint2* __restrict__ q, uint8_t* __restrict__ sf,
                                                      int64_t rb_q, const int32_t* __restrict__ pstart,
                                                      const int32_t* __restrict__ ends, int E) {
  constexpr int TPR = 32 * WPR;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = warp / WPR, t = threadIdx.x % TPR;
  const int64_t team0 = (int64_t)blockIdx.x * (8 / WPR) + team;
  const int64_t nteams = (int64_t)gridDim.x * (8 / WPR);
  const int64_t ncb = nvec / 16;  // 128-column scale blocks per row
  if (JAG && __ldg(pstart + E) == 0) return;  // offsets rejected: nothing is written
  int e = 0;
  for (int64_t r = team0; r < rows; r += nteams) {
    int64_t b = 0, pr = r;  // batch entry; the row's position in the scale layout
    if (JAG) {
      while (e < E - 1 && __ldg(ends + e) <= r) ++e;
      pr = __ldg(pstart + e) + (r - (e ? __ldg(ends + e - 1) : 0));
    } else {
      b = r / R;
      pr = r - b * R;
    }
    const uint4* xr = x + r * nvec;
    uint4 v[kMxRowVPL];
#pragma unroll
    for (int i = 0; i < kMxRowVPL; ++i) {
      const int c = t + TPR * i;
      v[i] = c < nvec ? ld_nc_v4(xr + c) : make_uint4(0, 0, 0, 0);
    }
    uint2* qr = q + r * nvec;
    uint8_t* srow = sf + (b * rb_q + (pr >> 7)) * ncb * 512 + (pr & 31) * 16 + ((pr >> 5) & 3) * 4;
#pragma unroll
    for (int i = 0; i < kMxRowVPL; ++i) {
      const int c = t + TPR * i;
      if (TPR * i >= nvec) break;  // uniform: nvec % 16 == 0 and every lane's c < nvec below it
      uint32_t m = absmax_fold(absmax_vec8(0u, v[i]));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const uint32_t code = mx_code<FMT>(m);
      const float inv = mx_inv(code);
      const int hb = lane & 16;
      const uint32_t word = __shfl_sync(0xffffffffu, code, hb) | (__shfl_sync(0xffffffffu, code, hb + 4) << 8) |
                            (__shfl_sync(0xffffffffu, code, hb + 8) << 16) |
                            (__shfl_sync(0xffffffffu, code, hb + 12) << 24);
      if (c < nvec) {
        uint2 o;
        o.x = mx_cast2<FMT>(v[i].x, inv) | (mx_cast2<FMT>(v[i].y, inv) << 16);
        o.y = mx_cast2<FMT>(v[i].z, inv) | (mx_cast2<FMT>(v[i].w, inv) << 16);
        qr[c] = o;
        if ((lane & 15) == 0) *reinterpret_cast<uint32_t*>(srow + (int64_t)(c / 16) * 512) = word;
      }
    }
  }
}

template <int FMT, int WPR, bool JAG>
int run_mx_rows(const MxArgs& a, int64_t rows, const Ctx& c) {
  auto kern = mx_rows_kernel<FMT, WPR, JAG>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
  const int64_t slots = (int64_t)c.sm_count * per_sm * (8 / WPR);  // teams resident at once
  const int64_t waves = ceil_div64(rows, slots);
  const int64_t teams = ceil_div64(rows, waves);
  kern<<<(unsigned)ceil_div64(teams, 8 / WPR), 256, 0, c.stream>>>(
      reinterpret_cast<const uint4*>(a.x), rows, a.R, (int)(a.C / 8), reinterpret_cast<uint2*>(a.q), a.sf, a.rb_q,
      a.pstart, a.ends, a.E);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

template <int FMT, bool JAG>
int dispatch_mx_rows(const MxArgs& a, int64_t rows, const Ctx& c) {
  const int nvec = (int)(a.C / 8);
  if (nvec <= 32 * kMxRowVPL) return run_mx_rows<FMT, 1, JAG>(a, rows, c);
  if (nvec <= 64 * kMxRowVPL) return run_mx_rows<FMT, 2, JAG>(a, rows, c);
  return run_mx_rows<FMT, 4, JAG>(a, rows, c);
}

template <int FMT, bool ROWS, bool COLS, bool JAG>
int run_mx_pipe(const MxArgs& a, int64_t grid_y, int64_t batches, const Ctx& c) {
  auto kern = mx_pipe_kernel<FMT, ROWS, COLS, JAG>;
  const int smem = kMpSmem + (JAG ? kMpMaxTiles * (int)sizeof(MpDesc) : 0);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return FP8_ERR_CUDA;
  const int64_t rows_total = JAG ? a.R : a.R * batches;
  if (rows_total > INT32_MAX || a.C > INT32_MAX) return FP8_ERR_UNSUPPORTED;  // TMA coordinates
  CUtensorMap tm;
  const uint64_t dims[2] = {(uint64_t)a.C, (uint64_t)rows_total};
  const uint64_t strides[1] = {(uint64_t)a.C * 2};
  const uint32_t box[2] = {64, kTile};
  const int rc = make_tmap(&tm, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != FP8_OK) return rc;
  const int64_t ncols = a.C / kTile, n_tiles = ncols * grid_y * batches;
  int64_t grid = n_tiles < c.sm_count ? n_tiles : c.sm_count;
  if (JAG && ceil_div64(n_tiles, grid) > kMpMaxTiles) grid = ceil_div64(n_tiles, kMpMaxTiles);  // descriptors fit
  if (grid > INT32_MAX) return FP8_ERR_UNSUPPORTED;
  kern<<<(unsigned)grid, kMpThreads, smem, c.stream>>>(tm, a, ncols, grid_y, n_tiles, c.status, c.wait_ns,
                                                       c.test_stall);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// The column-major output (with or without the row-major one) on the pipelined kernel; the
// row-major output alone on row teams while a row fits their registers.
template <int FMT, bool JAG>
int dispatch_layout(const MxArgs& a, int64_t grid_y, int64_t batches, const Ctx& c) {
  if (a.q && a.qt) return run_mx_pipe<FMT, true, true, JAG>(a, grid_y, batches, c);
  // the row-major output alone by row teams, for rows of up to 4 * 32 * 16 vectors of 8
  if (a.q && a.C / 8 <= 128 * kMxRowVPL) return dispatch_mx_rows<FMT, JAG>(a, a.R * batches, c);
  if (a.q) return run_mx_pipe<FMT, true, false, JAG>(a, grid_y, batches, c);
  return run_mx_pipe<FMT, false, true, JAG>(a, grid_y, batches, c);
}

}  // namespace

int64_t mx_scale_bytes(int64_t rows, int64_t k) {
  if (rows < 0 || k < 0 || k % 128) return -1;
  return (rows + 127) / 128 * 128 * (k / 32);
}

int launch_mx_quant(const void* x, int64_t batches, int64_t R, int64_t C, int fmt, void* q, void* sf, void* qt,
                    int64_t ld_t, void* sft, const int32_t* ends, int64_t E, int32_t* pstart_ws, const Ctx& c) {
  if (C % kTile || (!q && !qt)) return FP8_ERR_INVALID_ARG;
  if (ends && (E < 1 || E > kMaxSegments || batches != 1)) return FP8_ERR_UNSUPPORTED;
  MxArgs a = {};
  a.x = static_cast<const uint16_t*>(x);
  a.R = R;
  a.C = C;
  a.q = static_cast<uint8_t*>(q);
  a.sf = static_cast<uint8_t*>(sf);
  a.qt = static_cast<uint8_t*>(qt);
  a.ld_t = ld_t;
  a.sft = static_cast<uint8_t*>(sft);
  a.ends = ends;
  a.E = (int)E;
  if (R == 0 || C == 0 || batches == 0) return FP8_OK;
  if (ends) {
    // row-major scales and the column-major codes both live in the padded row space [0, P)
    a.rb_q = ld_t / kTile;
    a.pstart = pstart_ws;
    mx_pstart_kernel<<<1, 1024, 0, c.stream>>>(ends, (int)E, R, ld_t, pstart_ws, c.status);
    if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
    const int64_t grid_y = ld_t / kTile;
    return fmt == FP8_DT_E4M3 ? dispatch_layout<FP8_DT_E4M3, true>(a, grid_y, 1, c)
                              : dispatch_layout<FP8_DT_E5M2, true>(a, grid_y, 1, c);
  }
  a.rb_q = (R + kTile - 1) / kTile;
  const int64_t grid_y = (R + kTile - 1) / kTile;
  if (grid_y > 65535 || batches > 65535) return FP8_ERR_UNSUPPORTED;
  return fmt == FP8_DT_E4M3 ? dispatch_layout<FP8_DT_E4M3, false>(a, grid_y, batches, c)
                            : dispatch_layout<FP8_DT_E5M2, false>(a, grid_y, batches, c);
}

}  // namespace fp8lin
