// Fused decode FFN: the grouped gate|up (with SwiGLU) and the grouped down
// projection of decode-sized batches in ONE persistent tcgen05 kernel.
//
// Decode is bound by the bytes of the activated sub-experts' weights
// (METRO, "Balancing Activated Experts (not Tokens) for Memory-Bound MoE
// Serving", §1-2); each weight byte is read once per step.  Running the two
// projections as separate launches leaves a launch gap and an idle tail
// between them.  Here every CTA walks one list: all gate|up items first,
// then all down items.  A down item streams its first weight stages at once
// and only its activation loads wait for the gate|up items of its token chunk
// (a per-chunk completion counter, bounded wait), so the down weight stream
// overlaps the end of the gate|up phase (MoE-Prism, arXiv 2510.19366, §III-B1
// Eq. (1): A = SiLU(X Wg) * (X Wu), X' = A Wdown).
//
// Item shapes (weight-stationary, "swap AB"): 128 weight rows are the MMA M
// side and a unit's token chunk (<= 64 rows) the N side.
//   gate|up item: 64 gate rows over the matching 64 up rows, K = H;
//                 TMEM lanes 0-63 gate, 64-127 up; up warps hand their values
//                 to the gate warps through shared memory; act is bf16.
//   down item:    128 rows of Wdown, K = I_sub; y_perm is bf16.
// Each pipeline stage carries two 64-column sub-blocks (H and I_sub are
// multiples of 128).  Roles: warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer, warps 2-5 epilogue.  Every wait is bounded.
#include "gemm_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kBK = 64;
constexpr int kKsub = 2;                       // 64-column sub-blocks per stage
constexpr int kM = 128;
constexpr int kGU = 64;                        // neurons per gate|up item
constexpr int kTokBox = 16;
constexpr int kThreads = 192;
constexpr int kGatherThreads = 128;             // warps 6..9 of the row-gathering variant
constexpr int kQ = 4;                          // item queue depth
constexpr uint32_t kWSub = kM * kBK * 2;        // 16 KB per weight sub-block
constexpr uint32_t kW = kWSub * kKsub;          // 32 KB

// Token chunk (tokens per item: 64, or 16 for batches of at most 16 tokens,
// whose smaller token buffers leave room for more weight stages in flight)
// and ring depth.
template <int CHUNK, int STAGES>
struct FfnCfg {
  static constexpr int kChunk = CHUNK;
  static constexpr int kStages = STAGES;
  static constexpr uint32_t kTokSub = CHUNK * kBK * 2;  // per token sub-block
  static constexpr uint32_t kTok = kTokSub * kKsub;
  static constexpr uint32_t kStage = kW + kTok;
  static constexpr uint32_t kOffB = STAGES * kW;
  static constexpr uint32_t kOffBar = STAGES * kStage;
  static constexpr uint32_t kNumBars = 2 * STAGES + 5 + 2 * kQ;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffPrefix = kOffMisc + 16 + kQ * 4;
  static constexpr uint32_t kOffOffs = kOffPrefix + (kMaxGroups + 1) * 4;
  static constexpr uint32_t kOffX = (kOffOffs + (kMaxGroups + 1) * 4 + 15) / 16 * 16;
  static constexpr uint32_t kSmemBytes = kOffX + kGU * 17 * 4 + 1024;
  // two accumulator buffers of CHUNK columns, or of 2 * CHUNK when a down item
  // is two 128-row blocks (DPAIR: one block per half of the buffer)
  static constexpr uint32_t kTmemCols = 2 * CHUNK < 32 ? 32 : 2 * CHUNK;
  static constexpr uint32_t kTmemColsPair = 4 * CHUNK < 32 ? 32 : 4 * CHUNK;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct FParams {
  const int32_t* offsets;
  int n_groups;
  int H;
  int I;
  int gu_tiles;          // I / 64 gate|up items per token chunk
  int dn_tiles;          // down items per token chunk: H / 128, or H / 256 (DPAIR)
  __nv_bfloat16* act;    // [out_rows, I]
  __nv_bfloat16* y;      // [out_rows, H]
  int32_t* done;         // [m-tiles] gate|up items finished per chunk; zero at launch
  int32_t* work;         // next item number (dynamic schedule); zero at launch
  int32_t* split_cnt;    // [kFfnPartSlots / 2] arrivals of split gate|up items; zero at launch
  float* part;           // [kFfnPartSlots][kChunk][128] fp32 partial sums of split items
  long long out_rows;
  int32_t* status;
  uint32_t debug_flags;
  const uint4* gx;       // GATHER: gate|up token rows are gx[gtok[r]] (bf16 [*, H])
  const int32_t* gtok;
  int gx_rows;
};

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 1 on every one of the 128 epilogue threads iff `ok` is non-zero on all of
// them (named barrier 1 with an AND reduction).  The epilogue warps meet at
// named barriers inside an item, so they must leave the item loop together:
// a warp whose bounded wait gave up must not leave another waiting at one.
__device__ __forceinline__ int epilogue_all(int ok) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(ok)
      : "memory");
  return r;
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Item w of the launch: w < n_gu is a gate|up item (chunk mt, neuron block
// m, hidden-dimension split s of S), else a down item (chunk mt, row block m).
struct Item {
  bool gu;
  int mt, m, s;
};

__device__ __forceinline__ Item item_of(int w, int n_gu, int S, int gu_tiles, int dn_tiles) {
  Item it;
  it.gu = w < n_gu;
  if (it.gu) {
    const int r = w / S;
    it.s = w - r * S;
    it.mt = r / gu_tiles;
    it.m = r - it.mt * gu_tiles;
  } else {
    const int v = w - n_gu;
    it.s = 0;
    it.mt = v / dn_tiles;
    it.m = v - it.mt * dn_tiles;
  }
  return it;
}

// GATHER: four more warps copy the token rows of every gate|up stage straight
// from x (row r of the chunk = token gtok[row0 + r]) into the swizzled token
// buffer with cp.async, so no permuted copy of x is needed; they follow the
// item queue like the MMA and epilogue warps, arrive on every stage's `full`
// (copies for gate|up items, none for down items, whose activation rows come
// by TMA), and the producer then loads only weights for gate|up items.
template <int CHUNK, int STAGES, bool GATHER = false, bool DPAIR = false>
__global__ void __launch_bounds__(GATHER ? kThreads + kGatherThreads : kThreads, 1)
    decode_ffn_kernel(const __grid_constant__ CUtensorMap tmWgu,
                      const __grid_constant__ CUtensorMap tmX16,
                      const __grid_constant__ CUtensorMap tmX64,
                      const __grid_constant__ CUtensorMap tmWdn,
                      const __grid_constant__ CUtensorMap tmA16,
                      const __grid_constant__ CUtensorMap tmA64, const FParams p) {
  using Cfg = FfnCfg<CHUNK, STAGES>;
  constexpr int kChunk = Cfg::kChunk;
  constexpr int kStages = Cfg::kStages;
  constexpr uint32_t kTokSub = Cfg::kTokSub, kTok = Cfg::kTok, kOffB = Cfg::kOffB;
  constexpr uint32_t kOffBar = Cfg::kOffBar, kOffMisc = Cfg::kOffMisc;
  constexpr uint32_t kOffPrefix = Cfg::kOffPrefix, kOffOffs = Cfg::kOffOffs, kOffX = Cfg::kOffX;
  constexpr uint32_t kTmemCols = Cfg::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint64_t* q_full = mma_done + 1;
  uint64_t* q_empty = q_full + kQ;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* s_total = reinterpret_cast<int*>(smem + kOffMisc + 8);
  volatile int* s_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 12);
  volatile int* s_item = reinterpret_cast<volatile int*>(smem + kOffMisc + 16);
  int* s_prefix = reinterpret_cast<int*>(smem + kOffPrefix);
  int* s_offs = reinterpret_cast<int*>(smem + kOffOffs);
  float* s_xchg = reinterpret_cast<float*>(smem + kOffX);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // set-up that reads nothing upstream overlaps the previous launch's tail
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], GATHER ? 1 + kGatherThreads : 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 4);
    mbar_init(&tempty[1], 4);
    mbar_init(mma_done, 1);
    for (int q = 0; q < kQ; ++q) {
      mbar_init(&q_full[q], 1);
      // the MMA thread, the four epilogue warps (and the four gather warps)
      mbar_init(&q_empty[q], GATHER ? 9 : 5);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmWgu);
    tma_prefetch_desc(&tmX16);
    tma_prefetch_desc(&tmX64);
    tma_prefetch_desc(&tmWdn);
    tma_prefetch_desc(&tmA16);
    tma_prefetch_desc(&tmA64);
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, DPAIR ? Cfg::kTmemColsPair : kTmemCols);
    tmem_relinquish();
  }
  pdl_wait_and_trigger();
  if (warp == 2)
    build_tile_table<kChunk>(p.offsets, p.n_groups, 0, p.out_rows, s_prefix, s_offs, s_total,
                             p.status, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int n_mt = *s_total;
  const int KB_gu = p.H / (kBK * kKsub);
  // stages of a down item: 128 columns of K each, or 64 (DPAIR)
  const int KB_dn = DPAIR ? p.I / kBK : p.I / (kBK * kKsub);
  constexpr int acc_cols = DPAIR ? 2 * kChunk : kChunk;   // TMEM columns per accumulator buffer
  // Few gate|up items (small batches): split each over the hidden dimension
  // so that more SMs stream the weights; the last split to finish adds the
  // partial sums in split order and applies SwiGLU.
  const int n_gu1 = n_mt * p.gu_tiles;
  int S = 1;
  if (KB_gu % 2 == 0 && 2 * n_gu1 <= static_cast<int>(gridDim.x) && 2 * n_gu1 <= kFfnPartSlots)
    S = 2;
  if (KB_gu % 4 == 0 && 4 * n_gu1 <= static_cast<int>(gridDim.x) && 4 * n_gu1 <= kFfnPartSlots)
    S = 4;
  const int n_gu = n_gu1 * S;
  const int total_work = n_gu + n_mt * p.dn_tiles;
  const int KB_split = KB_gu / S;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      bool skip = (p.debug_flags & MOE_DEBUG_SKIP_FIRST_LOAD) != 0u;
      bool ok = true;
      // the first item of every CTA is its block index; later ones come
      // from the shared counter
      int w_next = static_cast<int>(blockIdx.x);
      for (int i = 0; ok; ++i) {
        const int slot = i % kQ;
        if (!mbar_wait(&q_empty[slot], ((i / kQ) & 1) ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        const int w = w_next < total_work ? w_next : -1;
        s_item[slot] = w;
        mbar_arrive(&q_full[slot]);
        if (w < 0) break;
        // the next item's number arrives while this one streams
        w_next = static_cast<int>(gridDim.x) + atomicAdd(p.work, 1);
        const Item it = item_of(w, n_gu, S, p.gu_tiles, p.dn_tiles);
        const Tile t = decode_tile<kChunk>(it.mt, 1, p.n_groups, s_prefix, s_offs);
        const int nb = (t.rows + kTokBox - 1) / kTokBox;
        const bool wide = nb > 2;
        const uint32_t tok_rows = wide ? 64u : static_cast<uint32_t>(nb * kTokBox);
        const bool gathered = GATHER && it.gu;   // token rows come from the gather warps
        const bool dpair = DPAIR && !it.gu;   // two weight blocks, one token sub-block
        const uint32_t bytes =
            gathered ? kW : kW + (dpair ? 1u : static_cast<uint32_t>(kKsub)) * tok_rows * kBK * 2;
        const int kb0 = it.gu ? it.s * KB_split : 0;
        const int kb1 = it.gu ? kb0 + KB_split : KB_dn;
        const CUtensorMap* mW = it.gu ? &tmWgu : &tmWdn;
        const CUtensorMap* mT = it.gu ? (wide ? &tmX64 : &tmX16) : (wide ? &tmA64 : &tmA16);
        const int wrow = it.gu ? t.g * 2 * p.I + it.m * kGU : t.g * p.H + it.m * (dpair ? 2 * kM : kM);
        auto weights = [&](uint8_t* sa, int kb) {
          if (dpair) {   // rows wrow.. and wrow + 128.. of the stage's 64 columns
            tma_load_2d(sa, mW, &full[stage], kb * kBK, wrow);
            tma_load_2d(sa + kWSub, mW, &full[stage], kb * kBK, wrow + kM);
            return;
          }
#pragma unroll
          for (int j = 0; j < kKsub; ++j) {
            const int kc = (kb * kKsub + j) * kBK;
            tma_load_2d(sa + j * kWSub, mW, &full[stage], kc, wrow);
            if (it.gu)  // the same 64 neurons' up rows fill the lower half
              tma_load_2d(sa + j * kWSub + kGU * kBK * 2, mW, &full[stage], kc, wrow + p.I);
          }
        };
        auto tokens = [&](uint8_t* sb, uint64_t* bar, int kb) {
#pragma unroll
          for (int j = 0; j < kKsub; ++j) {
            if (dpair && j > 0) break;
            const int kc = dpair ? kb * kBK : (kb * kKsub + j) * kBK;
            if (wide) {
              tma_load_2d(sb + j * kTokSub, mT, bar, kc, t.row0);
            } else {
              for (int b = 0; b < nb; ++b)
                tma_load_2d(sb + j * kTokSub + b * kTokBox * kBK * 2, mT, bar, kc,
                            t.row0 + b * kTokBox);
            }
          }
        };
        int kb = kb0;
        if (!it.gu) {
          // Down item: put the first weight stages in flight, then wait until
          // every gate|up item of this token chunk has stored its act rows.
          const int pre = kb1 - kb0 < kStages ? kb1 - kb0 : kStages;
          int st0 = stage;
          for (; kb < kb0 + pre; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&full[stage], bytes);
            weights(smem + stage * kW, kb);
            issued |= 1u << stage;
            issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          const uint64_t t0 = globaltimer();
          while (ld_acquire(p.done + it.mt) < p.gu_tiles) {
            if (*s_abort || globaltimer() - t0 > kWaitLimitNs) {
              ok = false;
              break;
            }
          }
          fence_proxy_async_global();
          // the token loads of the pre-issued stages (their full barriers
          // already expect these bytes)
          for (int i2 = 0; i2 < pre; ++i2) {
            const int s = (st0 + i2) % kStages;
            tokens(smem + kOffB + s * kTok, &full[s], kb0 + i2);
          }
          if (!ok) break;
        }
        for (; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          if (skip) {
            skip = false;  // test hook: the consumer of this slot must time out
          } else {
            mbar_expect_tx(&full[stage], bytes);
            weights(smem + stage * kW, kb);
            if (!gathered) tokens(smem + kOffB + stage * kTok, &full[stage], kb);
            issued |= 1u << stage;
            issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) fail(s_abort, p.status);
      for (int s = 0; s < kStages; ++s)
        if ((issued >> s) & 1u) mbar_wait(&full[s], (issued_par >> s) & 1u, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int slot = i % kQ;
        if (!mbar_wait(&q_full[slot], (i / kQ) & 1, s_abort)) {
          ok = false;
          break;
        }
        const int w = s_item[slot];
        mbar_arrive(&q_empty[slot]);
        if (w < 0) break;
        const Item it = item_of(w, n_gu, S, p.gu_tiles, p.dn_tiles);
        const Tile t = decode_tile<kChunk>(it.mt, 1, p.n_groups, s_prefix, s_offs);
        const int n = ((t.rows + 15) / 16) * 16;
        const uint32_t idesc = idesc_bf16_f32(kM, n);
        const int KB = it.gu ? KB_split : KB_dn;
        if (!mbar_wait(&tempty[acc], aphase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * acc_cols);
        const bool dpair = DPAIR && !it.gu;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(&full[stage], phase, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (dpair) {
            // weight blocks 0 and 1 of the stage against its one token
            // sub-block, into the two halves of the accumulator buffer
            const uint64_t b = sdesc_sw128(smem_u32(smem + kOffB + stage * kTok));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t a = sdesc_sw128(smem_u32(smem + stage * kW + h * kWSub));
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                umma_bf16(d + static_cast<uint32_t>(h * kChunk), a + 2u * k, b + 2u * k, idesc,
                          (kb | k) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < kKsub; ++j) {
              const uint64_t a = sdesc_sw128(smem_u32(smem + stage * kW + j * kWSub));
              const uint64_t b = sdesc_sw128(smem_u32(smem + kOffB + stage * kTok + j * kTokSub));
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                umma_bf16(d, a + 2u * k, b + 2u * k, idesc, (kb | j | k) != 0 ? 1u : 0u);
            }
          }
          umma_commit(&empty[stage]);
          if (++stage == kStages) {
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
      umma_commit(mma_done);
      mbar_wait(mma_done, 0u, nullptr);
    }
    __syncwarp();
  } else if (GATHER && warp >= 6) {
    // Row gather of gate|up items: thread g copies 16-byte chunk (g % 8) of
    // token rows g / 8 + 16 i (i < kChunk / 16) of both 64-column sub-blocks
    // of every stage; the chunk lands at chunk ^ (row % 8) of its 128-byte
    // row (the 128-byte swizzle of the TMA boxes it replaces).  A stage's
    // copies are one cp.async group; once a group is LAG groups old the
    // thread waits for it, orders it for the tensor cores' async-proxy reads
    // and arrives on that stage's `full`.  Down-item stages (no copies) are
    // arrived on at once.  Held-back arrivals are all made before a down item
    // and before the thread has to wait for its next item: the producer
    // publishes that item only after a down item's activations exist, which
    // may need these very stages.
    constexpr int LAG = kStages - 2;
    constexpr int kRowsPer = kChunk / 16;
    const int g = threadIdx.x - kThreads;
    const int chunk = g & 7, rg = g >> 3;
    const size_t nv = static_cast<size_t>(p.H) / 8;
    int stage = 0, astage = 0, pending = 0;
    uint32_t phase = 0;
    bool ok = true, bad = false;
    auto flush = [&]() {
      if (pending > 0) {
        asm volatile("cp.async.wait_all;" ::: "memory");
        fence_proxy_async_smem();
        for (; pending > 0; --pending) {
          mbar_arrive(&full[astage]);
          if (++astage == kStages) astage = 0;
        }
      }
    };
    for (int i = 0; ok; ++i) {
      const int slot = i % kQ;
      int avail = 1;
      if (lane == 0) avail = mbar_try_wait(&q_full[slot], (i / kQ) & 1) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, avail, 0)) flush();   // the producer may be waiting on them
      int got = 1;
      if (lane == 0) got = mbar_wait(&q_full[slot], (i / kQ) & 1, s_abort) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        ok = false;
        break;
      }
      int w = 0;
      if (lane == 0) {
        w = s_item[slot];
        mbar_arrive(&q_empty[slot]);
      }
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w < 0) break;
      const Item it = item_of(w, n_gu, S, p.gu_tiles, p.dn_tiles);
      const Tile t = decode_tile<kChunk>(it.mt, 1, p.n_groups, s_prefix, s_offs);
      const uint4* src[kRowsPer];
#pragma unroll
      for (int j = 0; j < kRowsPer; ++j) {
        const int r = rg + 16 * j;
        int tok = -1;
        if (it.gu && r < t.rows) {
          tok = __ldg(p.gtok + t.row0 + r);
          if (tok < 0 || tok >= p.gx_rows) {
            bad = true;
            tok = -1;
          }
        }
        src[j] = tok >= 0 ? p.gx + static_cast<size_t>(tok) * nv + chunk : nullptr;
      }
      if (!it.gu) {
        flush();
        for (int kb = 0; kb < KB_dn; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive(&full[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        astage = stage;
        continue;
      }
      const int kb0 = it.s * KB_split;
      const int kb1 = kb0 + KB_split;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        const uint32_t sb = smem_u32(smem + kOffB + stage * kTok);
#pragma unroll
        for (int sub = 0; sub < kKsub; ++sub)
#pragma unroll
          for (int j = 0; j < kRowsPer; ++j) {
            const int r = rg + 16 * j;
            if (src[j] != nullptr)
              asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                               sb + sub * kTokSub + r * 128 + ((chunk ^ (r & 7)) << 4)),
                           "l"(src[j] + (kb * kKsub + sub) * (kBK / 8))
                           : "memory");
          }
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (++pending > LAG) {
          asm volatile("cp.async.wait_group %0;" ::"n"(LAG) : "memory");
          fence_proxy_async_smem();
          mbar_arrive(&full[astage]);
          if (++astage == kStages) astage = 0;
          --pending;
        }
        if (++stage == kStages) {
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
        if (++astage == kStages) astage = 0;
      }
    } else if (lane == 0) {
      fail(s_abort, p.status);
    }
    if (bad) report(p.status, MOE_ERR_BAD_INDEX);
  } else {
    const int q = warp & 3;
    const int r_in = q * 32 + lane;
    int acc = 0;
    uint32_t aphase = 0;
    for (int i = 0;; ++i) {
      const int slot = i % kQ;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&q_full[slot], (i / kQ) & 1, s_abort) ? 1 : 0;
      ok = epilogue_all(__shfl_sync(0xffffffffu, ok, 0));
      if (!ok) {
        if (lane == 0) fail(s_abort, p.status);
        break;
      }
      int w = 0;
      if (lane == 0) {
        w = s_item[slot];
        mbar_arrive(&q_empty[slot]);
      }
      w = __shfl_sync(0xffffffffu, w, 0);
      if (w < 0) break;
      const Item it = item_of(w, n_gu, S, p.gu_tiles, p.dn_tiles);
      const Tile t = decode_tile<kChunk>(it.mt, 1, p.n_groups, s_prefix, s_offs);
      if (lane == 0) ok = mbar_wait(&tfull[acc], aphase, s_abort) ? 1 : 0;
      ok = epilogue_all(__shfl_sync(0xffffffffu, ok, 0));
      if (!ok) {
        if (lane == 0) fail(s_abort, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(acc * acc_cols);
      if (it.gu && S == 1) {
        const bool is_gate = q < 2;
        const int nl = (q & 1) * 32 + lane;
        const int col = it.m * kGU + nl;
        for (int c0 = 0; c0 < t.rows; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tb + c0, v);
          tmem_ld_wait();
          if (!is_gate) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) s_xchg[nl * 17 + cc] = __uint_as_float(v[cc]);
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (is_gate) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
              const long long r = static_cast<long long>(t.row0) + c0 + cc;
              if (c0 + cc < t.rows && r < p.out_rows)
                p.act[r * p.I + col] = __float2bfloat16_rn(silu_f(__uint_as_float(v[cc])) *
                                                           s_xchg[nl * 17 + cc]);
            }
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");
        }
        // publish: this chunk's act columns [m*64, m*64+64) are stored
        fence_proxy_async_global();
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (warp == 2 && lane == 0) atomicAdd(p.done + it.mt, 1);
      } else if (it.gu) {
        // split item: fp32 partial [token][row] to this split's slot; the
        // last split of the item to arrive finishes it
        const int item = it.mt * p.gu_tiles + it.m;
        float* mine = p.part + static_cast<size_t>(item * S + it.s) * (kChunk * kM);
        for (int c0 = 0; c0 < t.rows; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tb + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int cc = 0; cc < 16; ++cc)
            if (c0 + cc < t.rows) mine[(c0 + cc) * kM + r_in] = __uint_as_float(v[cc]);
        }
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (warp == 2 && lane == 0) *s_flag = atomicAdd(p.split_cnt + item, 1);
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (*s_flag == S - 1) {
          __threadfence();
          if (q < 2) {
            const float* base = p.part + static_cast<size_t>(item * S) * (kChunk * kM);
            const int col = it.m * kGU + r_in;
            for (int c = 0; c < t.rows; ++c) {
              float g = 0.f, u = 0.f;
              for (int s2 = 0; s2 < S; ++s2) {
                g += __ldcg(base + static_cast<size_t>(s2) * (kChunk * kM) + c * kM + r_in);
                u += __ldcg(base + static_cast<size_t>(s2) * (kChunk * kM) + c * kM + kGU + r_in);
              }
              const long long r = static_cast<long long>(t.row0) + c;
              if (r < p.out_rows) p.act[r * p.I + col] = __float2bfloat16_rn(silu_f(g) * u);
            }
          }
          fence_proxy_async_global();
          __threadfence();
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (warp == 2 && lane == 0) atomicAdd(p.done + it.mt, 1);
        }
      } else {
        // down: one 128-row block, or two (DPAIR: rows h * 128 + r_in)
#pragma unroll 1
        for (int h = 0; h < (DPAIR ? 2 : 1); ++h) {
          const int col = it.m * (DPAIR ? 2 * kM : kM) + h * kM + r_in;
          for (int c0 = 0; c0 < t.rows; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tb + static_cast<uint32_t>(h * kChunk) + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
              const long long r = static_cast<long long>(t.row0) + c0 + cc;
              if (c0 + cc < t.rows && r < p.out_rows)
                p.y[r * p.H + col] = __float2bfloat16_rn(__uint_as_float(v[cc]));
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, DPAIR ? Cfg::kTmemColsPair : kTmemCols);
  }
}

}  // namespace

bool decode_ffn_supports(int H, int I_sub) { return H % 128 == 0 && I_sub % 128 == 0; }

cudaError_t launch_decode_ffn(const DecodeFfnArgs& a, cudaStream_t s) {
  if (a.x_rows <= 0 || a.rows <= 0) return cudaSuccess;
  CUtensorMap wgu, x16, x64, wdn, a16, a64;
  const int E_r = a.n_groups;
  // with the row gather the x_perm maps are unused; they then describe x
  const void* xt = a.gather_x != nullptr ? a.gather_x : a.x_perm;
  const long long xt_rows = a.gather_x != nullptr ? a.gather_rows : a.x_rows;
  if (!make_tmap_bf16(&wgu, a.w_gate_up, static_cast<long long>(E_r) * 2 * a.I, a.H, kGU) ||
      !make_tmap_bf16(&x16, xt, xt_rows, a.H, kTokBox) ||
      !make_tmap_bf16(&x64, xt, xt_rows, a.H, 64) ||
      !make_tmap_bf16(&wdn, a.w_down, static_cast<long long>(E_r) * a.H, a.I, kM) ||
      !make_tmap_bf16(&a16, a.act, a.rows, a.I, kTokBox) ||
      !make_tmap_bf16(&a64, a.act, a.rows, a.I, 64))
    return cudaErrorInvalidValue;
  FParams p;
  p.offsets = a.offsets;
  p.n_groups = E_r;
  p.H = a.H;
  p.I = a.I;
  p.gu_tiles = a.I / kGU;
  p.dn_tiles = a.H / kM;
  p.act = static_cast<__nv_bfloat16*>(a.act);
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.done = a.done;
  p.work = a.work;
  p.split_cnt = a.split_cnt;
  p.part = a.part;
  p.out_rows = a.rows;
  p.status = a.status;
  p.debug_flags = a.debug_flags;
  p.gx = static_cast<const uint4*>(a.gather_x);
  p.gtok = a.gather_tok;
  p.gx_rows = a.gather_rows;
  const bool gather = a.gather_x != nullptr;
  if (gather && a.gather_tok == nullptr) return cudaErrorInvalidValue;
  if (a.chunk == 16) {
    using Cfg = FfnCfg<16, 6>;
    if (gather) {
      static bool attr_done[64] = {false};
      cudaError_t e = set_smem_once(decode_ffn_kernel<16, 6, true>,
                                    static_cast<int>(Cfg::kSmemBytes), attr_done);
      if (e != cudaSuccess) return e;
      return launch_pdl(decode_ffn_kernel<16, 6, true>, dim3(a.sm_count),
                        dim3(kThreads + kGatherThreads), Cfg::kSmemBytes, s, wgu, x16, x64, wdn,
                        a16, a64, p);
    }
    static bool attr_done[64] = {false};
    cudaError_t e = set_smem_once(decode_ffn_kernel<16, 6>, static_cast<int>(Cfg::kSmemBytes),
                                  attr_done);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_ffn_kernel<16, 6>, dim3(a.sm_count), dim3(kThreads),
                      Cfg::kSmemBytes, s, wgu, x16, x64, wdn, a16, a64, p);
  }
  using Cfg = FfnCfg<64, 4>;
  // Small I with 64-token chunks: down items of two 128-row blocks (half as
  // many items, each streaming twice the weights through the same 32 KB
  // stages).  Same-box A/B, Qwen3-30B-A3B-shaped decode (I_sub 384): T = 64
  // 197.4 -> 186.8 us, T = 256 222.3 -> 212.0, T = 1024 238.2 -> 231.7; with
  // 16-token chunks (T <= 16) the halved item count costs more than it saves
  // (T = 1 28.6 -> 32.4 us, T = 8 74.2 -> 76.1), so those keep one block per
  // item.  A template parameter: the other variants keep their code and
  // registers.
  const bool dpair = a.I <= 1024 && a.H % (2 * kM) == 0;
  if (dpair) p.dn_tiles = a.H / (2 * kM);
  auto go = [&](auto kern, int threads) -> cudaError_t {
    return launch_pdl(kern, dim3(a.sm_count), dim3(threads), Cfg::kSmemBytes, s, wgu, x16, x64,
                      wdn, a16, a64, p);
  };
  if (gather) {
    if (dpair) {
      static bool attr_done[64] = {false};
      cudaError_t e = set_smem_once(decode_ffn_kernel<64, 4, true, true>,
                                    static_cast<int>(Cfg::kSmemBytes), attr_done);
      if (e != cudaSuccess) return e;
      return go(decode_ffn_kernel<64, 4, true, true>, kThreads + kGatherThreads);
    }
    static bool attr_done[64] = {false};
    cudaError_t e = set_smem_once(decode_ffn_kernel<64, 4, true>,
                                  static_cast<int>(Cfg::kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
    return go(decode_ffn_kernel<64, 4, true>, kThreads + kGatherThreads);
  }
  if (dpair) {
    static bool attr_done[64] = {false};
    cudaError_t e = set_smem_once(decode_ffn_kernel<64, 4, false, true>,
                                  static_cast<int>(Cfg::kSmemBytes), attr_done);
    if (e != cudaSuccess) return e;
    return go(decode_ffn_kernel<64, 4, false, true>, kThreads);
  }
  static bool attr_done[64] = {false};
  cudaError_t e = set_smem_once(decode_ffn_kernel<64, 4>, static_cast<int>(Cfg::kSmemBytes),
                                attr_done);
  if (e != cudaSuccess) return e;
  return go(decode_ffn_kernel<64, 4>, kThreads);
}

}  // namespace moe
