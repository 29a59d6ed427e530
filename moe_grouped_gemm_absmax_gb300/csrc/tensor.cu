// Tensorwise FP8 quantization with the tensor partly held on chip between its two reads (sm_103a).
//
// Recipe: "FP8 Training: Quantization, Autograd, Torchao", section 2 "The quantization math".
// Fusion: "FP8 training on AMD GPUs with TorchTitan and TorchAO", "Triton Kernel Optimization",
// Level 1 (one kernel per quantization, the row- and column-major outputs from one read of each
// element in the cast) and Level 3 (relaxed atomics for the amax).
//
// The scale needs the amax of the whole tensor, so every element is read twice. One cooperative
// launch, one CTA per SM, tiles of 128 rows x 64 columns dealt round-robin:
//   pass 1: a producer warp streams the CTA's tiles through a ring of 8 shared-memory slots by
//           TMA (128 KB in flight per SM); 8 warps fold |x| and release each slot. The last 8
//           tiles of every CTA are never overwritten: they stay on chip (19 MB over 152 SMs), and
//           the tiles read just before them are the newest lines in L2 (8 slots timed faster
//           than 6, 10 or 12);
//   barrier: the CTA's maximum goes to the workspace's amax word (relaxed atomic), the CTA counts
//           itself on the barrier word (release) and waits, bounded, until all have (acquire);
//   pass 2: the tiles in reverse order: the slots' own tiles first, then each freed slot is
//           refilled with the next older tile (from L2 while it is still there); each warp casts
//           32 rows of a tile (a lane per column pair), writes its row-major 32 x 64 box and its
//           column-major 64 x 32 box into shared memory and stores both by TMA.
// A wait that runs out sets FP8_DEV_TIMEOUT; the CTA drains its loads and stores and leaves.
#include "common.cuh"
#include "internal.h"

namespace fp8lin {

namespace {

constexpr int kTsRows = 128, kTsCols = 64;
constexpr int kTsTileBytes = kTsRows * kTsCols * 2;  // 16 KB of bf16, 128-byte swizzled rows
constexpr int kTsSlots = 8;
constexpr int kTsWarps = 8;                          // two groups of 4: group g casts tiles j = g mod 2
constexpr int kTsThreads = 32 * (kTsWarps + 1);      // + the producer warp
constexpr int kTsBox = 64 * 32;                      // one warp's box of codes (either layout)
constexpr uint64_t kTsDrainNs = 2000000000ull;       // fixed bound: loads in flight before exit

struct TsShared {
  uint64_t full[kTsSlots];   // the slot holds its tile (TMA bytes, or present from pass 1)
  uint64_t empty[kTsSlots];  // the 4 warps of the tile's group are done with the slot
  uint32_t red[kTsWarps];
  float s32;
  int ok;
  int abort;
};
constexpr size_t kTsSmem = 1024 + (size_t)kTsSlots * kTsTileBytes + 2 * kTsWarps * kTsBox + sizeof(TsShared);

template <int FMT>
__global__ void __launch_bounds__(kTsThreads, 1)
    quant_tensor_stash_kernel(const __grid_constant__ CUtensorMap tm_in, const __grid_constant__ CUtensorMap tm_q,
                              const __grid_constant__ CUtensorMap tm_qt, int64_t R, int64_t C, uint32_t* ws,
                              float* inv, int has_q, int has_qt, int32_t* status, uint64_t wait_ns, int test_stall,
                              const __grid_constant__ ScaleTab tab) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* slots = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* boxes = slots + kTsSlots * kTsTileBytes;
  TsShared& S = *reinterpret_cast<TsShared*>(boxes + 2 * kTsWarps * kTsBox);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t tcols = ceil_div64(C, kTsCols), ntiles = ceil_div64(R, kTsRows) * tcols;
  const int64_t cnt = (int64_t)blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto tile_rc = [&](int64_t k, int32_t* r0, int32_t* c0) {  // the CTA's k-th tile
    const int64_t t = blockIdx.x + k * (int64_t)gridDim.x;
    *r0 = (int32_t)((t / tcols) * kTsRows);
    *c0 = (int32_t)((t % tcols) * kTsCols);
  };
  auto init_barriers = [&]() {
    for (int s = 0; s < kTsSlots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 4);
    }
    fence_mbar_init();
  };
  if (tid == 0) {
    init_barriers();
    S.abort = 0;
    tma_prefetch_desc(&tm_in);
  }
  __syncthreads();
  volatile int* abort = &S.abort;
  auto fail = [&]() {
    if (!*abort) {
      *abort = 1;
      set_status(status, FP8_DEV_TIMEOUT);
    }
  };
  const int grp = warp >> 2, wq = warp & 3;  // cast warps: group, 32-row quarter of the tile
  // this lane's column pair within a 128-byte swizzled tile row r: chunk lane / 4, word lane % 4
  auto word_at = [&](const uint8_t* tile, int r) {
    return *reinterpret_cast<const uint32_t*>(tile + r * 128 + ((((uint32_t)lane >> 2) ^ (uint32_t)(r & 7)) << 4) +
                                              ((lane & 3) << 2));
  };

  // ==================================== pass 1: amax ====================================
  if (warp == kTsWarps) {
    if (lane == 0) {
      int64_t k = 0;
      for (; k < cnt; ++k) {
        const int s = (int)(k % kTsSlots);
        if (!mbar_wait(&S.empty[s], (uint32_t)(((k / kTsSlots) & 1) ^ 1), abort, wait_ns)) {
          fail();
          break;
        }
        int32_t r0, c0;
        tile_rc(k, &r0, &c0);
        // the tiles that stay in their slots need no L2 copy; the others are read again from L2
        const uint64_t pol = k + kTsSlots < cnt ? l2_evict_last() : l2_evict_first();
        mbar_arrive_expect_tx(&S.full[s], kTsTileBytes);
        tma_load_2d_hint(slots + s * kTsTileBytes, &tm_in, &S.full[s], c0, r0, pol);
      }
      for (int64_t j = k > kTsSlots ? k - kTsSlots : 0; j < k; ++j)  // loads in flight land before exit
        mbar_wait(&S.full[j % kTsSlots], (uint32_t)((j / kTsSlots) & 1), nullptr, kTsDrainNs);
    }
  } else {
    uint32_t acc = 0;
    for (int64_t k = grp; k < cnt; k += 2) {
      const int s = (int)(k % kTsSlots);
      if (!__all_sync(0xffffffffu, mbar_wait(&S.full[s], (uint32_t)((k / kTsSlots) & 1), abort, wait_ns))) {
        if (lane == 0) fail();
        break;
      }
      const uint8_t* tile = slots + s * kTsTileBytes;
#pragma unroll
      for (int r = 0; r < 32; ++r) acc = absmax2(acc, word_at(tile, 32 * wq + r));
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
    }
    acc = __reduce_max_sync(0xffffffffu, absmax_fold(acc));
    if (lane == 0) S.red[warp] = acc;
  }
  __syncthreads();
  // ==================== the grid barrier, then the scale from the table ====================
  if (tid == 0) {
    bool ok = !*abort;
    if (ok) {
      uint32_t m = 0;
      for (int w = 0; w < kTsWarps; ++w) m = max(m, S.red[w]);
      if (m) red_max_relaxed(ws, m);
      red_add_release_gpu(ws + 1, 1u);
      // the failure-detection test hook waits for one arrival more than there are CTAs
      ok = wait_count_geq(ws + 1, gridDim.x + (test_stall ? 1u : 0u), wait_ns);
      if (!ok) fail();
    }
    const Scale sc = tab_scale(tab, ld_relaxed_gpu(ws));
    S.s32 = sc.s32;
    S.ok = ok;
    if (blockIdx.x == 0 && ok) *inv = sc.inv32;
    if (ok) {  // every load of pass 1 was consumed: fresh barriers for pass 2
      for (int s = 0; s < kTsSlots; ++s) {
        mbar_inval(&S.full[s]);
        mbar_inval(&S.empty[s]);
      }
      init_barriers();
    }
  }
  __syncthreads();
  if (!S.ok) return;
  const float s32 = S.s32;

  // ============================ pass 2: the cast, newest tile first ============================
  // Sequence j handles the CTA's tile k = cnt - 1 - j in slot k % 8; the first 8 are in their
  // slots already, each later one is loaded into the slot the tile 8 steps earlier freed.
  if (warp == kTsWarps) {
    if (lane == 0) {
      int64_t j = 0;
      for (; j < cnt; ++j) {
        const int64_t k = cnt - 1 - j;
        const int s = (int)(k % kTsSlots);
        const int64_t u = j / kTsSlots;  // the slot's use in this pass
        if (u == 0) {
          mbar_arrive(&S.full[s]);  // present since pass 1
          continue;
        }
        if (!mbar_wait(&S.empty[s], (uint32_t)((u & 1) ^ 1), abort, wait_ns)) {
          fail();
          break;
        }
        int32_t r0, c0;
        tile_rc(k, &r0, &c0);
        mbar_arrive_expect_tx(&S.full[s], kTsTileBytes);
        tma_load_2d_hint(slots + s * kTsTileBytes, &tm_in, &S.full[s], c0, r0, l2_evict_first());
      }
      for (int64_t i = j > kTsSlots ? j - kTsSlots : kTsSlots; i < j; ++i)  // loads in flight land before exit
        mbar_wait(&S.full[(cnt - 1 - i) % kTsSlots], (uint32_t)((i / kTsSlots) & 1), nullptr, kTsDrainNs);
    }
  } else {
    const uint64_t out_pol = l2_evict_first();
    uint8_t* bq = boxes + warp * 2 * kTsBox;  // row-major box [32 rows][64 codes]
    uint8_t* bt = bq + kTsBox;                // column-major box [64 columns][32 codes]
    const float2 s2 = make_float2(s32, s32);
    for (int64_t j = grp; j < cnt; j += 2) {
      const int64_t k = cnt - 1 - j;
      const int s = (int)(k % kTsSlots);
      if (!__all_sync(0xffffffffu, mbar_wait(&S.full[s], (uint32_t)((j / kTsSlots) & 1), abort, wait_ns))) {
        if (lane == 0) fail();
        break;
      }
      const uint8_t* tile = slots + s * kTsTileBytes;
      uint32_t w[32];
#pragma unroll
      for (int r = 0; r < 32; ++r) w[r] = word_at(tile, 32 * wq + r);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);
      int32_t r0, c0;
      tile_rc(k, &r0, &c0);
      const int32_t row0 = r0 + 32 * wq;
      if (row0 >= R) continue;  // rows past the tensor: nothing to store
      // column 2 l: the low halves; column 2 l + 1: the high halves
      uint32_t olo[8], ohi[8], pr[32];
#pragma unroll
      for (int r = 0; r < 32; r += 4) {
        const float2 l01 = fmul2_rn(make_float2(__uint_as_float(w[r] << 16), __uint_as_float(w[r + 1] << 16)), s2);
        const float2 l23 = fmul2_rn(make_float2(__uint_as_float(w[r + 2] << 16), __uint_as_float(w[r + 3] << 16)), s2);
        const float2 h01 = fmul2_rn(make_float2(__uint_as_float(w[r] & 0xFFFF0000u), __uint_as_float(w[r + 1] & 0xFFFF0000u)), s2);
        const float2 h23 = fmul2_rn(make_float2(__uint_as_float(w[r + 2] & 0xFFFF0000u), __uint_as_float(w[r + 3] & 0xFFFF0000u)), s2);
        const uint32_t a = cvt_fp8x2<FMT>(l01.x, l01.y), b = cvt_fp8x2<FMT>(l23.x, l23.y);
        const uint32_t c = cvt_fp8x2<FMT>(h01.x, h01.y), d = cvt_fp8x2<FMT>(h23.x, h23.y);
        olo[r / 4] = a | (b << 16);
        ohi[r / 4] = c | (d << 16);
        // row-major: the pair (column 2 l, column 2 l + 1) of rows r .. r + 3
        pr[r] = __byte_perm(a, c, 0x0040);
        pr[r + 1] = __byte_perm(a, c, 0x0051);
        pr[r + 2] = __byte_perm(b, d, 0x0040);
        pr[r + 3] = __byte_perm(b, d, 0x0051);
      }
      if (lane == 0) bulk_wait_read_all();  // the previous tile's stores have read the boxes
      __syncwarp();
      if (has_q) {
#pragma unroll
        for (int r = 0; r < 32; ++r) *reinterpret_cast<uint16_t*>(bq + r * 64 + 2 * lane) = (uint16_t)pr[r];
      }
      if (has_qt) {
        uint8_t* dst = bt + lane * 64;  // rows 2 l and 2 l + 1 of the box: 32 codes each
        *reinterpret_cast<uint4*>(dst) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
        *reinterpret_cast<uint4*>(dst + 16) = make_uint4(olo[4], olo[5], olo[6], olo[7]);
        *reinterpret_cast<uint4*>(dst + 32) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
        *reinterpret_cast<uint4*>(dst + 48) = make_uint4(ohi[4], ohi[5], ohi[6], ohi[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (has_q) tma_store_2d_hint(&tm_q, bq, c0, row0, out_pol);
        if (has_qt) tma_store_2d_hint(&tm_qt, bt, row0, c0, out_pol);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_all();
  }
  __syncthreads();
}

}  // namespace

// The stash kernel's conditions: the row-major codes leave by TMA (their row stride, C bytes,
// a multiple of 16) and the column-major ones too (R bytes, which the entry point already requires).
bool tensor_stash_ok(int64_t R, int64_t C, bool has_q, bool has_qt) {
  return R > 0 && C > 0 && R <= INT32_MAX && C <= INT32_MAX && (!has_q || C % 16 == 0) && (!has_qt || R % 16 == 0);
}

int launch_quant_tensor_stash(const void* x, int64_t R, int64_t C, int fmt, void* q, void* qt, float* inv,
                              uint32_t* ws, const Ctx& c) {
  // ws[0]: the amax word, ws[1]: the barrier count; both start at zero
  if (cudaMemsetAsync(ws, 0, 2 * sizeof(uint32_t), c.stream) != cudaSuccess) return FP8_ERR_CUDA;
  CUtensorMap tin, tq, tqt;
  int rc;
  {
    const uint64_t dims[2] = {(uint64_t)C, (uint64_t)R};
    const uint64_t strides[1] = {(uint64_t)C * 2};
    const uint32_t box[2] = {kTsCols, kTsRows};
    rc = make_tmap(&tin, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != FP8_OK) return rc;
  }
  tq = tin;
  tqt = tin;
  if (q) {
    const uint64_t dims[2] = {(uint64_t)C, (uint64_t)R};
    const uint64_t strides[1] = {(uint64_t)C};
    const uint32_t box[2] = {64, 32};  // 32 rows x 64 codes
    rc = make_tmap(&tq, q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != FP8_OK) return rc;
  }
  if (qt) {
    const uint64_t dims[2] = {(uint64_t)R, (uint64_t)C};
    const uint64_t strides[1] = {(uint64_t)R};
    const uint32_t box[2] = {32, 64};  // 64 columns x 32 codes
    rc = make_tmap(&tqt, qt, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != FP8_OK) return rc;
  }
  const int64_t ntiles = ceil_div64(R, kTsRows) * ceil_div64(C, kTsCols);
  const unsigned grid = (unsigned)(ntiles < c.sm_count ? ntiles : c.sm_count);
  auto kern = fmt == FP8_DT_E4M3 ? quant_tensor_stash_kernel<FP8_DT_E4M3> : quant_tensor_stash_kernel<FP8_DT_E5M2>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTsSmem) != cudaSuccess)
    return FP8_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: they meet at the grid barrier
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTsThreads);
  cfg.dynamicSmemBytes = kTsSmem;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tin, tq, tqt, R, C, ws, inv, q ? 1 : 0, qt ? 1 : 0, c.status, c.wait_ns,
                         c.test_stall, scale_tab(fmt)) != cudaSuccess)
    return FP8_ERR_CUDA;
  return FP8_OK;
}

}  // namespace fp8lin
