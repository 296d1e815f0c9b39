// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by
// TMA, for the expert FFN of the k-aware MoE layer.
//
//   D[r, n] = sum_k A[r, k] * B[b_row(g, n), k]      r in the rows of group g
//
// Groups are routing units (rows of unit u are offsets[u] .. offsets[u+1]),
// or one dense group (router logits, shared expert).  Three epilogues:
//   EPI_SWIGLU  the B tile is a gate slab and the matching up slab of one
//               sub-expert; act = SiLU(gate) * up, stored bf16
//               (MoE-Prism, arXiv 2510.19366, §III-B1 Eq. (1))
//   EPI_BF16    plain bf16 store (down projection, X' = A Wdown)
//   EPI_F32     fp32 store plus a per-expert bias (router logits, §III-B2)
//
// Structure: persistent CTAs (one per SM), 6 warps.
//   warp 0      TMA producer: one elected thread streams A and B k-blocks
//               (64 bf16 = 128 B wide, 128-byte swizzle) into a STAGES-deep
//               shared-memory ring, completion counted on `full` mbarriers
//   warp 1      allocates TMEM; one elected thread issues tcgen05.mma
//               (M = 128, N = BN_MMA, K = 16) into one of two fp32 TMEM
//               accumulators, and commits to `empty` (ring slot free) and
//               `tfull` (accumulator ready) mbarriers
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane TMEM quadrant (one
//               output row per thread), math; a warp whose 32 rows all belong
//               to the tile's unit stages each 32 x 64 bf16 block in shared
//               memory and writes it with one TMA store, a partial slab uses
//               masked 16-byte stores; then release the accumulator on `tempty`
// Work items are (m-tile, n-tile) pairs, m-tile major, handed out
// round-robin; the m-tile -> (unit, first row) map is rebuilt in shared
// memory from `offsets` at kernel start, so no host sync is needed.
// Every wait is bounded (MOE_ERR_DEVICE_TIMEOUT), loads in flight are
// drained and TMEM is freed before the CTA exits.
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_common.cuh"
#include "moe_internal.h"

namespace moe {

bool make_tmap_bf16(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows);
bool make_tmap_f32(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows);

namespace {

constexpr int BM = kTileRows;
constexpr int BK = 64;
constexpr int kThreads = 192;
constexpr int kGatherThreads = 128;   // warps 6..9 of the row-gathering variant
constexpr uint32_t kABytes = BM * BK * 2;

struct KParams {
  const int32_t* offsets;
  int n_groups;
  int dense_rows;
  int K;
  int n_tiles;       // n-tiles per group
  int bn_out;        // output columns per n-tile
  int b_group_rows;  // rows of B per group
  int b_up_offset;   // SWIGLU: rows between a gate row and its up row
  void* out;
  long long ld_out;
  long long out_rows;
  int out_cols;      // EPI_F32: valid output columns
  const uint4* gx;           // GATHER: A rows are x[gtok[r]] (bf16 [*, K]), 16-byte vectors
  const int32_t* gtok;       // GATHER: token of every permuted row
  int gx_rows;               // GATHER: rows of x (tokens outside are reported and skipped)
  int k_splits;      // EPI_F32: the hidden dimension split S ways, partial sums to
  long long split_stride;  // out + s * split_stride (elements); 1: no split
  const float* bias;
  int bias_div;
  int32_t* status;
  uint32_t debug_flags;
  int f32_tma;       // EPI_F32: full 32-row slabs leave through TMA stores (tmOut: fp32
                     //   [S * out_rows, ld_out], 32 x 32 boxes); 0: per-thread stores only
};

template <int BN_MMA, int STAGES>
struct Cfg {
  static constexpr uint32_t kBBytes = BN_MMA * BK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = (2 * BN_MMA <= 32)    ? 32
                                        : (2 * BN_MMA <= 64)  ? 64
                                        : (2 * BN_MMA <= 128) ? 128
                                        : (2 * BN_MMA <= 256) ? 256
                                                              : 512;
  static constexpr uint32_t kOffA = 0;
  static constexpr uint32_t kOffB = STAGES * kABytes;
  static constexpr uint32_t kOffStage = STAGES * kStageBytes;  // 4 epilogue buffers
  static constexpr uint32_t kOffBar = kOffStage + 4 * kStageRowsBytes;
  static constexpr uint32_t kNumBars = 2 * STAGES + 5;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffPrefix = kOffMisc + 16;
  static constexpr uint32_t kOffOffs = kOffPrefix + (kMaxGroups + 1) * 4;
  static constexpr uint32_t kSmemUsed = kOffOffs + (kMaxGroups + 1) * 4;
  static constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // 1024-B alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(BN_MMA % 16 == 0 && BN_MMA >= 16 && BN_MMA <= 256, "tcgen05 N for M = 128");
};

// GATHER: four more warps copy the A rows of every k-block straight from x
// (row r of the tile is token gtok[row0 + r]) into the swizzled A stage with
// cp.async, so no permuted copy of x is materialised; the producer then loads
// only B.
template <int BN_MMA, int EPI, int STAGES, bool GATHER = false>
__global__ void __launch_bounds__(GATHER ? kThreads + kGatherThreads : kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmOut, const KParams p) {
  using C = Cfg<BN_MMA, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int* s_total = reinterpret_cast<int*>(smem + C::kOffMisc + 8);
  int* s_prefix = reinterpret_cast<int*>(smem + C::kOffPrefix);
  int* s_offs = reinterpret_cast<int*>(smem + C::kOffOffs);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // set-up that reads nothing written upstream runs before the grid
  // dependency wait, overlapping the previous kernel's tail
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // GATHER: the producer's arrive (B bytes) plus one cp.async arrive per gather thread
      mbar_init(&full[s], GATHER ? 1 + kGatherThreads : 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 4);
    mbar_init(&tempty[1], 4);
    mbar_init(done, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    if (!GATHER) tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (EPI != EPI_F32 || p.f32_tma) tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  pdl_wait_and_trigger();
  if (warp == 2) build_tile_table(p.offsets, p.n_groups, p.dense_rows, p.out_rows, s_prefix, s_offs,
                                  s_total, p.status, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  // EPI_F32 may split K: n-tile index nt * S + s, split s covers k-blocks
  // [s * KB / S, (s + 1) * KB / S)
  const int S = EPI == EPI_F32 ? p.k_splits : 1;
  const int n_tiles_eff = p.n_tiles * S;
  const int total_work = *s_total * n_tiles_eff;
  const int KB = p.K / BK / S;
  const int G = p.offsets == nullptr ? 1 : p.n_groups;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_par = 0;
      bool skip = (p.debug_flags & MOE_DEBUG_SKIP_FIRST_LOAD) != 0u;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < total_work; w += gridDim.x) {
        const Tile t = decode_tile(w, n_tiles_eff, G, s_prefix, s_offs);
        const int split = t.nt % S, nt = t.nt / S;
        const int b_row = t.g * p.b_group_rows + nt * p.bn_out;
        for (int kb = split * KB; kb < (split + 1) * KB; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          if (skip) {
            skip = false;  // test hook: the consumer of this slot must time out
          } else {
            uint8_t* sa = smem + C::kOffA + stage * kABytes;
            uint8_t* sb = smem + C::kOffB + stage * C::kBBytes;
            mbar_expect_tx(&full[stage], GATHER ? C::kBBytes : C::kStageBytes);
            if (!GATHER) tma_load_2d(sa, &tmA, &full[stage], kb * BK, t.row0);
            if (EPI == EPI_SWIGLU) {
              tma_load_2d(sb, &tmB, &full[stage], kb * BK, b_row);
              tma_load_2d(sb + (BN_MMA / 2) * BK * 2, &tmB, &full[stage], kb * BK,
                          b_row + p.b_up_offset);
            } else {
              tma_load_2d(sb, &tmB, &full[stage], kb * BK, b_row);
            }
            issued |= 1u << stage;
            issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) fail(s_abort, p.status);
      // every load issued here must land before the CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait(&full[s], (issued_par >> s) & 1u, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN_MMA);
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < total_work; w += gridDim.x) {
        if (!mbar_wait(&tempty[acc], aphase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * BN_MMA);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(smem_u32(smem + C::kOffA + stage * kABytes));
          const uint64_t bd = sdesc_sw128(smem_u32(smem + C::kOffB + stage * C::kBBytes));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d, ad + 2u * k, bd + 2u * k, idesc, (kb | k) != 0 ? 1u : 0u);  // kb from 0
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          aphase ^= 1u;
        }
      }
      if (!ok) fail(s_abort, p.status);
      // all MMAs issued here must be complete before TMEM is released
      umma_commit(done);
      mbar_wait(done, 0u, nullptr);
    }
    __syncwarp();
  } else if (GATHER && warp >= 6) {
    // A-row gather: thread g copies 16-byte chunk (g % 8) of rows g / 8 + 16 i
    // (i < 8) of every k-block; the chunk lands at chunk ^ (row % 8) of its
    // 128-byte row (the 128-byte swizzle the MMA descriptors expect).  The
    // copies of a stage are one cp.async group; once a group is LAG groups
    // old the thread waits for it, orders it for the tensor cores' async-proxy
    // reads (fence.proxy.async) and arrives on that stage's `full` barrier.
    // LAG = STAGES - 2 keeps that arrival independent of the MMA's progress on
    // the stage just before, so the tensor pipe is never held by it.
    constexpr int LAG = STAGES - 2;
    const int g = threadIdx.x - kThreads;
    const int chunk = g & 7, rg = g >> 3;
    const uint32_t dst_off = static_cast<uint32_t>(rg * 128 + ((chunk ^ (rg & 7)) << 4));
    const size_t nv = static_cast<size_t>(p.K) / 8;
    int stage = 0, astage = 0, pending = 0;
    uint32_t phase = 0;
    bool ok = true, bad = false;
    // the token indices of an item are loaded one item ahead, so the first
    // copies of an item do not wait for them
    auto load_tokens = [&](int w, int (&tk)[8]) {
      const Tile t = decode_tile(w, n_tiles_eff, G, s_prefix, s_offs);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rg + 16 * i;
        tk[i] = r < t.rows ? __ldg(p.gtok + t.row0 + r) : -1;
      }
    };
    int tk[8];
    if (static_cast<int>(blockIdx.x) < total_work) load_tokens(blockIdx.x, tk);
    for (int w = blockIdx.x; ok && w < total_work; w += gridDim.x) {
      const uint4* src[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int tok = tk[i];
        if (tok != -1 && (tok < 0 || tok >= p.gx_rows)) {
          bad = true;
          tok = -1;
        }
        src[i] = tok >= 0 ? p.gx + static_cast<size_t>(tok) * nv + chunk : nullptr;
      }
      if (w + static_cast<int>(gridDim.x) < total_work) load_tokens(w + gridDim.x, tk);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(smem + C::kOffA + stage * kABytes) + dst_off;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (src[i] != nullptr)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa + i * 16 * 128),
                         "l"(src[i] + kb * (BK / 8))
                         : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (++pending > LAG) {
          asm volatile("cp.async.wait_group %0;" ::"n"(LAG) : "memory");
          fence_proxy_async_smem();
          mbar_arrive(&full[astage]);
          if (++astage == STAGES) astage = 0;
          --pending;
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (ok) {
      fence_proxy_async_smem();
      for (; pending > 0; --pending) {
        mbar_arrive(&full[astage]);
        if (++astage == STAGES) astage = 0;
      }
    } else {
      fail(s_abort, p.status);
    }
    if (bad) report(p.status, MOE_ERR_BAD_INDEX);
  } else {
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r_in = q * 32 + lane;
    uint8_t* sbuf = smem + C::kOffStage + q * kStageRowsBytes;
    int acc = 0;
    uint32_t aphase = 0;
    for (int w = blockIdx.x; w < total_work; w += gridDim.x) {
      Tile t = decode_tile(w, n_tiles_eff, G, s_prefix, s_offs);
      const int split = t.nt % S;
      t.nt /= S;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], aphase, s_abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) fail(s_abort, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN_MMA);
      const long long grow = static_cast<long long>(t.row0) + r_in;
      const bool valid = r_in < t.rows && grow < p.out_rows;
      if (EPI != EPI_F32) {
        // every row of this warp's slab belongs to the tile's unit
        const bool full_slab = q * 32 + 32 <= t.rows &&
                               static_cast<long long>(t.row0) + q * 32 + 32 <= p.out_rows;
        const int col0 = t.nt * p.bn_out;
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + grow * p.ld_out + col0;
        constexpr int kCols = EPI == EPI_SWIGLU ? BN_MMA / 2 : BN_MMA;  // outputs per row
#pragma unroll 1
        for (int c = 0; c < kCols; c += 32) {
          uint32_t pk[16];
          if (EPI == EPI_SWIGLU) {
            uint32_t gv[32], uv[32];
            tmem_ld32(tbase + c, gv);
            tmem_ld32(tbase + BN_MMA / 2 + c, uv);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a0 = silu_f(__uint_as_float(gv[2 * i])) * __uint_as_float(uv[2 * i]);
              const float a1 =
                  silu_f(__uint_as_float(gv[2 * i + 1])) * __uint_as_float(uv[2 * i + 1]);
              pk[i] = pack_bf16x2(a0, a1);
            }
          } else {
            uint32_t v[32];
            tmem_ld32(tbase + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          }
          if (full_slab) {
            if ((c & 32) == 0) {  // first half of a 64-column block: buffer free?
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
            }
            stage_row_32(sbuf, lane, (c & 32) >> 3, pk);
            if ((c & 32) != 0) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmOut, sbuf, col0 + c - 32, t.row0 + q * 32);
                bulk_commit();
              }
            }
          } else if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
      } else {
        const int col0 = t.nt * p.bn_out;
        float* orow = static_cast<float*>(p.out) + split * p.split_stride + grow * p.ld_out + col0;
        // a warp whose 32 rows are all real writes each 32 x 32 fp32 block
        // through shared memory with one TMA store (128-byte swizzle, as for
        // bf16); other rows use per-thread stores
        const bool full_slab = p.f32_tma && q * 32 + 32 <= t.rows &&
                               static_cast<long long>(t.row0) + q * 32 + 32 <= p.out_rows &&
                               col0 + BN_MMA <= p.out_cols;
#pragma unroll 1
        for (int c = 0; c < BN_MMA; c += 32) {
          uint32_t v[32];
          tmem_ld32(tbase + c, v);
          tmem_ld_wait();
          if (full_slab) {
            uint32_t lo[16], hi[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float a = __uint_as_float(v[i]), b = __uint_as_float(v[16 + i]);
              if (p.bias != nullptr) {
                a += p.bias[(col0 + c + i) / p.bias_div];
                b += p.bias[(col0 + c + 16 + i) / p.bias_div];
              }
              lo[i] = __float_as_uint(a);
              hi[i] = __float_as_uint(b);
            }
            if (lane == 0) bulk_wait_read_all();   // the previous block has left the buffer
            __syncwarp();
            stage_row_32(sbuf, lane, 0, lo);
            stage_row_32(sbuf, lane, 4, hi);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmOut, sbuf, col0 + c,
                           static_cast<int>(split * p.out_rows + t.row0 + q * 32));
              bulk_commit();
            }
            continue;
          }
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const int col = col0 + c + i;
              if (col + 4 <= p.out_cols) {
                float4 f;
                f.x = __uint_as_float(v[i]);
                f.y = __uint_as_float(v[i + 1]);
                f.z = __uint_as_float(v[i + 2]);
                f.w = __uint_as_float(v[i + 3]);
                if (p.bias != nullptr) {
                  f.x += p.bias[(col + 0) / p.bias_div];
                  f.y += p.bias[(col + 1) / p.bias_div];
                  f.z += p.bias[(col + 2) / p.bias_div];
                  f.w += p.bias[(col + 3) / p.bias_div];
                }
                *reinterpret_cast<float4*>(orow + c + i) = f;
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_all();  // stores done before the CTA (and its smem) goes
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

template <int BN_MMA, int EPI, int STAGES, bool GATHER = false>
cudaError_t run_gemm(const GemmArgs& g, cudaStream_t s) {
  using C = Cfg<BN_MMA, STAGES>;
  const int box_b = EPI == EPI_SWIGLU ? BN_MMA / 2 : BN_MMA;  // output columns per n-tile
  CUtensorMap ta, tb, to;
  if (GATHER) {
    if (g.gather_x == nullptr || g.gather_tok == nullptr) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&ta, g.gather_x, 1, g.K, 1)) return cudaErrorInvalidValue;  // unused
  } else if (!make_tmap_bf16(&ta, g.a, g.a_rows, g.K, BM)) {
    return cudaErrorInvalidValue;
  }
  if (!make_tmap_bf16(&tb, g.b, g.b_rows, g.K, box_b)) return cudaErrorInvalidValue;
  bool f32_tma = false;
  if (EPI == EPI_F32) {
    // fp32 [S * out_rows, ld_out] when the split slices are contiguous
    const int S = g.k_splits > 1 ? g.k_splits : 1;
    const bool contiguous = S == 1 || g.split_stride == g.out_rows * g.ld_out;
    f32_tma = contiguous &&
              make_tmap_f32(&to, g.out, g.out_rows * S, static_cast<int>(g.ld_out), 32);
    if (!f32_tma) to = tb;  // unused
  } else if (!make_tmap_bf16(&to, g.out, g.out_rows, static_cast<int>(g.ld_out), 32)) {
    return cudaErrorInvalidValue;
  }
  KParams kp;
  kp.offsets = g.offsets;
  kp.n_groups = g.offsets == nullptr ? 1 : g.n_groups;
  kp.dense_rows = g.dense_rows;
  kp.K = g.K;
  kp.bn_out = box_b;
  kp.n_tiles = (g.n_out + box_b - 1) / box_b;
  kp.b_group_rows = g.b_group_rows;
  kp.b_up_offset = EPI == EPI_SWIGLU ? g.n_out : 0;
  kp.out = g.out;
  kp.ld_out = g.ld_out;
  kp.out_rows = g.out_rows;
  kp.out_cols = g.n_out;
  kp.gx = static_cast<const uint4*>(g.gather_x);
  kp.gtok = g.gather_tok;
  kp.gx_rows = g.gather_rows;
  kp.k_splits = EPI == EPI_F32 && g.k_splits > 1 ? g.k_splits : 1;
  kp.split_stride = g.split_stride;
  if (g.K % (BK * kp.k_splits) != 0) return cudaErrorInvalidValue;
  kp.bias = kp.k_splits > 1 ? nullptr : g.bias;
  kp.bias_div = g.bias_div > 0 ? g.bias_div : 1;
  kp.status = g.status;
  kp.debug_flags = g.debug_flags;
  kp.f32_tma = f32_tma ? 1 : 0;
  long long m_tiles;
  if (g.offsets == nullptr)
    m_tiles = (g.dense_rows + BM - 1) / BM;
  else
    m_tiles = (g.max_rows_hint + BM - 1) / BM + g.n_groups;
  const long long work = m_tiles * kp.n_tiles * kp.k_splits;
  if (work <= 0) return cudaSuccess;
  const int grid = static_cast<int>(work < g.sm_count ? work : g.sm_count);
  auto kern = grouped_gemm_kernel<BN_MMA, EPI, STAGES, GATHER>;
  // The shared-memory opt-in is set once per device, so that launches made
  // while a stream is being captured into a CUDA graph issue no other call.
  static bool attr_done[64] = {false};
  cudaError_t e = set_smem_once(kern, static_cast<int>(C::kSmemBytes), attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(GATHER ? kThreads + kGatherThreads : kThreads),
                    C::kSmemBytes, s, ta, tb, to, kp);
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Encoded tensor maps, keyed by everything that goes into them, so that a
// call on tensors seen before skips the encoding (host time of the small
// decode calls); host memory only.  64 sets of 4 ways: a key goes to the set
// its hashed fields pick (every field mixed into the set index, so the 16-
// and 64-row boxes of one tensor do not evict each other), and a new key
// replaces the set's ways in turn.
namespace {
struct TmapKey {
  const void* base;
  long long rows;
  int cols, box_rows, elem;
  bool operator==(const TmapKey& o) const {
    return base == o.base && rows == o.rows && cols == o.cols && box_rows == o.box_rows &&
           elem == o.elem;
  }
};
constexpr int kTmapSets = 64, kTmapWays = 4;
struct TmapCache {
  std::mutex mu;
  TmapKey key[kTmapSets][kTmapWays] = {};
  CUtensorMap map[kTmapSets][kTmapWays];
  bool used[kTmapSets][kTmapWays] = {};
  int next[kTmapSets] = {};
};
TmapCache& tmap_cache() {
  static TmapCache c;
  return c;
}
// 64-bit finaliser (xor-shift and odd-constant multiplies) of a running hash
uint64_t tmap_mix(uint64_t h) {
  h ^= h >> 33;
  h *= 0xff51afd7ed558ccdull;
  h ^= h >> 33;
  h *= 0xc4ceb9fe1a85ec53ull;
  h ^= h >> 33;
  return h;
}
int tmap_set(const TmapKey& k) {
  uint64_t h = tmap_mix(static_cast<uint64_t>(reinterpret_cast<uintptr_t>(k.base)));
  h = tmap_mix(h ^ static_cast<uint64_t>(k.rows));
  h = tmap_mix(h ^ (static_cast<uint64_t>(static_cast<uint32_t>(k.cols)) << 32 ^
                    static_cast<uint64_t>(static_cast<uint32_t>(k.box_rows)) << 8 ^
                    static_cast<uint64_t>(static_cast<uint32_t>(k.elem))));
  return static_cast<int>(h % kTmapSets);
}
bool tmap_lookup(const TmapKey& k, CUtensorMap* m) {
  TmapCache& c = tmap_cache();
  const int i = tmap_set(k);
  std::lock_guard<std::mutex> g(c.mu);
  for (int w = 0; w < kTmapWays; ++w)
    if (c.used[i][w] && c.key[i][w] == k) {
      *m = c.map[i][w];
      return true;
    }
  return false;
}
void tmap_store(const TmapKey& k, const CUtensorMap& m) {
  TmapCache& c = tmap_cache();
  const int i = tmap_set(k);
  std::lock_guard<std::mutex> g(c.mu);
  for (int w = 0; w < kTmapWays; ++w)
    if (c.used[i][w] && c.key[i][w] == k) return;
  const int w = c.next[i];
  c.next[i] = (w + 1) % kTmapWays;
  c.key[i][w] = k;
  c.map[i][w] = m;
  c.used[i][w] = true;
}
}  // namespace

// bf16 [rows, cols] row-major, box = 64 columns x box_rows rows, 128-B swizzle.
bool make_tmap_bf16(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows) {
  const TmapKey key{base, rows, cols, box_rows, 2};
  if (rows > 0 && tmap_lookup(key, m)) return true;
  auto fn = encode_fn();
  if (fn == nullptr || rows <= 0) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  tmap_store(key, *m);
  return true;
}

// fp32 [rows, cols] row-major, boxes of 32 columns (128 bytes) x box_rows.
bool make_tmap_f32(CUtensorMap* m, const void* base, long long rows, int cols, int box_rows) {
  const TmapKey key{base, rows, cols, box_rows, 4};
  if (rows > 0 && tmap_lookup(key, m)) return true;
  auto fn = encode_fn();
  if (fn == nullptr || rows <= 0 || cols % 32 != 0 ||
      (reinterpret_cast<uintptr_t>(base) & 15u) != 0)
    return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  cuuint32_t box[2] = {32u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  tmap_store(key, *m);
  return true;
}

bool gemm_supports_f32_router(int E_r) { return E_r == 64 || E_r == 128 || E_r == 256; }

void router_gemm_shape(int T, int H, int E_r, int* bn, int* splits) {
  *bn = T < 4096 ? 64 : E_r;
  const long long base = static_cast<long long>((T + BM - 1) / BM) * (E_r / *bn);
  const int KB = H / BK;
  int S = 1;
  while (S < 8 && base * S * 2 <= 128 && KB % (S * 2) == 0) S *= 2;
  *splits = S;
}

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t s) {
  // CTA pairs stage a third fewer bytes per SM and k-block.  Routed GEMMs run
  // on them when the caller asks (force_pair; the pair kernel tiles each
  // unit's remainder of <= 128 rows with M = 128, so padding stays as with
  // single CTAs); dense GEMMs use pairs when the 256-row padding allows it.
  if (gemm_pair_supports(g.epi, g.n_out)) {
    bool pair = g.force_pair && g.offsets != nullptr;
    if (g.offsets == nullptr) {
      const long long p = (g.dense_rows + 255) / 256, t = (g.dense_rows + 127) / 128;
      pair = 86 * p <= 50 * t;  // 256 p rows at ~0.86 the cost of 128 t rows
    }
    if (pair) return launch_gemm_pair(g, s);
  }
  switch (g.epi) {
    case EPI_SWIGLU:
      if (g.gather_x != nullptr) {
        if (g.n_out % 128 == 0) return run_gemm<256, EPI_SWIGLU, 4, true>(g, s);
        return run_gemm<128, EPI_SWIGLU, 6, true>(g, s);
      }
      if (g.n_out % 128 == 0) return run_gemm<256, EPI_SWIGLU, 4>(g, s);
      return run_gemm<128, EPI_SWIGLU, 6>(g, s);
    case EPI_BF16:
      if (g.n_out % 256 == 0) return run_gemm<256, EPI_BF16, 4>(g, s);
      if (g.n_out % 128 == 0) return run_gemm<128, EPI_BF16, 6>(g, s);
      return run_gemm<64, EPI_BF16, 8>(g, s);
    case EPI_F32: {
      const int bn = g.bn_hint > 0 && g.bn_hint < g.n_out ? g.bn_hint : g.n_out;
      if (g.n_out % bn != 0) return cudaErrorInvalidValue;
      if (bn == 256) return run_gemm<256, EPI_F32, 4>(g, s);
      if (bn == 128) return run_gemm<128, EPI_F32, 6>(g, s);
      if (bn == 64) return run_gemm<64, EPI_F32, 8>(g, s);
      return cudaErrorInvalidValue;
    }
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
