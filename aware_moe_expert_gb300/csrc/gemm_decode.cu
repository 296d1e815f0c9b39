// Decode-shaped grouped GEMM ("swap AB"): when every routing unit holds only
// a few token rows, the weights are the 128-row tcgen05 M operand and the
// unit's tokens the small N operand (16..64), so each activated sub-expert's
// weights stream from HBM once per step while the tensor cores do no padded
// work on the weight side.  Decode is bound by the bytes of the activated
// experts' weights (MoE-Prism, arXiv 2510.19366, §II-A: work is linear in the
// routed assignments; METRO, "Balancing Activated Experts (not Tokens) for
// Memory-Bound MoE Serving", §1: decode time follows activated experts).
//
//   gate|up  D_g[n, c] = sum_k Wg_u[n, k] x_c[k],  D_u likewise, n in a
//            128-neuron slice; act[c, n] = SiLU(D_g) * D_u   (§III-B1 Eq. (1))
//   down     D[h, c] = sum_k Wd_u[h, k] act_c[k], h in a 128-row slice of H
//
// Work items are (token chunk of one unit (<= 64 rows), weight slice, K
// split).  The split count S is chosen on the device from the real number of
// items so that the persistent grid runs close to whole waves; with S > 1 the
// kernel writes fp32 partial sums, and split_swiglu_kernel (gate|up: adds
// the splits, then SiLU * up) or split_sum_kernel (down) adds them in split
// order, so the result does not depend on scheduling.
//
// Roles as in the prefill kernel: warp 0 TMA producer, warp 1 TMEM owner and
// MMA issuer, warps 2-5 epilogue (TMEM lane = weight row = output column).
#include "gemm_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kBK = 64;           // columns of one 128-byte swizzled sub-block
constexpr int kM = 128;           // weight rows per item (MMA M)
constexpr int kGU = 64;           // gate|up: neurons per item (64 gate rows over 64 up rows)
constexpr int kTokBox = 16;       // token rows per TMA box
constexpr int kThreads = 192;
constexpr uint32_t kWBytes = kM * kBK * 2;  // one weight sub-block: 16 KB
constexpr uint32_t kTmemCols = 512;         // 2 accumulator slots

struct DParams {
  const int32_t* offsets;
  int n_groups;
  int K;
  int m_tiles;          // weight slices per unit
  int w_group_rows;     // rows of the weight tensor per unit
  int w_up_offset;      // gate|up: rows from a gate row to its up row
  int n_out;            // output columns (gate|up: I_sub, down: H)
  void* out;            // bf16 [out_rows, n_out]
  float* partial;       // fp32 [max_split][out_rows][w * n_out], w = 2 (gate|up) or 1
  int32_t* split_word;  // receives the chosen S
  long long out_rows;
  int max_split;
  int32_t* status;
  uint32_t debug_flags;
  float item_bytes;     // weight bytes of one unsplit item
  float total_scale;    // 1 / (HBM bytes per ns) for the whole grid
};

// GATE_UP: two weight tiles (gate, up) per stage; CHUNK: tokens per item
// (MMA N <= CHUNK); KSUB: 64-column sub-blocks per pipeline stage.
template <bool GATE_UP, int STAGES, int CHUNK, int KSUB>
struct DCfg {
  static constexpr uint32_t kW = kWBytes * KSUB;                        // one weight tile
  static constexpr uint32_t kA = kW;  // gate|up: 64 gate rows stacked over 64 up rows
  static constexpr uint32_t kTokSub = CHUNK * kBK * 2;                  // tokens, one sub-block
  static constexpr uint32_t kTokBytes = kTokSub * KSUB;
  static constexpr uint32_t kSlot = CHUNK;                              // TMEM columns per slot
  static constexpr uint32_t kStage = kA + kTokBytes;
  static constexpr uint32_t kOffB = STAGES * kA;
  static constexpr uint32_t kOffBar = STAGES * kStage;
  static constexpr uint32_t kNumBars = 2 * STAGES + 5;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kOffPrefix = kOffMisc + 16;
  static constexpr uint32_t kOffOffs = kOffPrefix + (kMaxGroups + 1) * 4;
  static constexpr uint32_t kOffX = (kOffOffs + (kMaxGroups + 1) * 4 + 15) / 16 * 16;
  static constexpr uint32_t kXBytes = GATE_UP ? kGU * 17 * 4 : 0;  // up values for gate warps
  static constexpr uint32_t kSmemBytes = kOffX + kXBytes + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(2 * kSlot <= kTmemCols, "two accumulator slots in TMEM");
  static_assert(CHUNK % 16 == 0 && CHUNK <= 256 && CHUNK >= 64, "tcgen05 N for M = 128");
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

// Split count for `items1` unsplit items of `item_bytes` weight bytes on a
// grid of G CTAs.  Estimated time of split S: the larger of the whole-grid
// HBM time and the per-CTA streaming time of the busiest CTA (waves x bytes
// per split item at the rate one SM sustains), plus a reduction launch when
// S > 1.  The smallest S within 3% of the best estimate wins.
__device__ __forceinline__ int choose_split(int items1, int G, int max_split, int KB,
                                            float item_bytes, float hbm_ns_per_byte) {
  if (items1 <= 0) return 1;
  constexpr float kSmBytesPerNs = 100.f;   // one SM streaming alone, ~100 GB/s
  constexpr float kReduceNs = 3000.f;      // extra launch + partial traffic
  const float total_ns = static_cast<float>(items1) * item_bytes * hbm_ns_per_byte;
  const int smax = min(max_split, KB);
  float t[9];
  float best = 3.4e38f;
  for (int s = 1; s <= smax && s <= 8; ++s) {
    const long long waves = (static_cast<long long>(items1) * s + G - 1) / G;
    const float per_cta = static_cast<float>(waves) * item_bytes / s / kSmBytesPerNs;
    t[s] = fmaxf(total_ns, per_cta) + (s > 1 ? kReduceNs : 0.f);
    best = fminf(best, t[s]);
  }
  for (int s = 1; s <= smax && s <= 8; ++s)
    if (t[s] <= best * 1.03f) return s;
  return 1;
}

template <bool GATE_UP, int STAGES, int CHUNK, int KSUB>
__global__ void __launch_bounds__(kThreads, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmX64, const DParams p) {
  using C = DCfg<GATE_UP, STAGES, CHUNK, KSUB>;
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
  float* s_xchg = reinterpret_cast<float*>(smem + C::kOffX);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // set-up that reads nothing written upstream runs before the grid
  // dependency wait, overlapping the previous kernel's tail
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
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
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmX64);
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  pdl_wait_and_trigger();
  if (warp == 2)
    build_tile_table<CHUNK>(p.offsets, p.n_groups, 0, p.out_rows, s_prefix, s_offs, s_total,
                             p.status, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const int KB = p.K / (kBK * KSUB);
  const int items1 = *s_total * p.m_tiles;
  const int S = choose_split(items1, gridDim.x, p.max_split, KB, p.item_bytes, p.total_scale);
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.split_word != nullptr) *p.split_word = S;
  const int per_mt = p.m_tiles * S;
  const int total_work = items1 * S;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_par = 0;
      bool skip = (p.debug_flags & MOE_DEBUG_SKIP_FIRST_LOAD) != 0u;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < total_work; w += gridDim.x) {
        const int mt = w / per_mt;
        const int rem = w - mt * per_mt;
        const int m = rem / S, s = rem - (rem / S) * S;
        const Tile t = decode_tile<CHUNK>(mt, 1, p.n_groups, s_prefix, s_offs);
        // token rows: up to two 16-row boxes, else 64-row boxes, per sub-block
        const int nb = (t.rows + kTokBox - 1) / kTokBox;
        const bool wide = nb > 2;
        const int nb64 = (t.rows + 63) / 64;
        const uint32_t tok_rows = wide ? 64u * nb64 : static_cast<uint32_t>(nb * kTokBox);
        const uint32_t bytes = C::kA + KSUB * tok_rows * kBK * 2;
        const int wrow = t.g * p.w_group_rows + m * (GATE_UP ? kGU : kM);
        const int kb0 = s * KB / S, kb1 = (s + 1) * KB / S;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort)) {
            ok = false;
            break;
          }
          if (skip) {
            skip = false;  // test hook: the consumer of this slot must time out
          } else {
            uint8_t* sa = smem + stage * C::kA;
            uint8_t* sb = smem + C::kOffB + stage * C::kTokBytes;
            mbar_expect_tx(&full[stage], bytes);
#pragma unroll
            for (int j = 0; j < KSUB; ++j) {
              const int kc = (kb * KSUB + j) * kBK;
              tma_load_2d(sa + j * kWBytes, &tmW, &full[stage], kc, wrow);
              if (GATE_UP)  // up rows of the same 64 neurons fill the lower half of the tile
                tma_load_2d(sa + j * kWBytes + kGU * kBK * 2, &tmW, &full[stage], kc,
                            wrow + p.w_up_offset);
              if (wide) {
                for (int b = 0; b < nb64; ++b)
                  tma_load_2d(sb + j * C::kTokSub + b * 64 * kBK * 2, &tmX64, &full[stage], kc,
                              t.row0 + b * 64);
              } else {
                for (int b = 0; b < nb; ++b)
                  tma_load_2d(sb + j * C::kTokSub + b * kTokBox * kBK * 2, &tmX, &full[stage], kc,
                              t.row0 + b * kTokBox);
              }
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
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) mbar_wait(&full[s], (issued_par >> s) & 1u, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < total_work; w += gridDim.x) {
        const int mt = w / per_mt;
        const int rem = w - mt * per_mt;
        const int s = rem - (rem / S) * S;
        const Tile t = decode_tile<CHUNK>(mt, 1, p.n_groups, s_prefix, s_offs);
        const int n = ((t.rows + 15) / 16) * 16;
        const uint32_t idesc = idesc_bf16_f32(kM, n);
        const int kb0 = s * KB / S, kb1 = (s + 1) * KB / S;
        if (!mbar_wait(&tempty[acc], aphase ^ 1u, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dg = tmem_base + static_cast<uint32_t>(acc) * C::kSlot;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int j = 0; j < KSUB; ++j) {
            const uint64_t ag = sdesc_sw128(smem_u32(smem + stage * C::kA + j * kWBytes));
            const uint64_t bx =
                sdesc_sw128(smem_u32(smem + C::kOffB + stage * C::kTokBytes + j * C::kTokSub));
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              const uint32_t accum = (kb != kb0 || j != 0 || k != 0) ? 1u : 0u;
              umma_bf16(dg, ag + 2u * k, bx + 2u * k, idesc, accum);
            }
          }
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
      umma_commit(done);
      mbar_wait(done, 0u, nullptr);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int r_in = q * 32 + lane;  // weight row inside the slice = TMEM lane
    int acc = 0;
    uint32_t aphase = 0;
    for (int w = blockIdx.x; w < total_work; w += gridDim.x) {
      const int mt = w / per_mt;
      const int rem = w - mt * per_mt;
      const int m = rem / S, s = rem - (rem / S) * S;
      const Tile t = decode_tile<CHUNK>(mt, 1, p.n_groups, s_prefix, s_offs);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], aphase, s_abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) fail(s_abort, p.status);
        break;
      }
      tc_fence_after();
      const uint32_t tg = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(acc) * C::kSlot;
      if (GATE_UP) {
        // TMEM lanes 0-63 hold the gate rows, 64-127 the up rows of the same
        // 64 neurons: warps of quadrants 2-3 hand their up values to the
        // gate warps (quadrants 0-1) through shared memory.
        const bool is_gate = q < 2;
        const int nl = (q & 1) * 32 + lane;
        const int col = m * kGU + nl;
        for (int c0 = 0; c0 < t.rows; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tg + c0, v);
          tmem_ld_wait();
          if (S > 1) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
              const long long r = static_cast<long long>(t.row0) + c0 + cc;
              if (c0 + cc < t.rows && r < p.out_rows)
                p.partial[(static_cast<long long>(s) * p.out_rows + r) * 2 * p.n_out +
                          (is_gate ? 0 : p.n_out) + col] = __uint_as_float(v[cc]);
            }
          } else {
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
                  static_cast<__nv_bfloat16*>(p.out)[r * p.n_out + col] = __float2bfloat16_rn(
                      silu_f(__uint_as_float(v[cc])) * s_xchg[nl * 17 + cc]);
              }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
          }
        }
      } else {
        const int col = m * kM + r_in;  // output column of this thread
        for (int c0 = 0; c0 < t.rows; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tg + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) {
            const long long r = static_cast<long long>(t.row0) + c0 + cc;
            if (c0 + cc < t.rows && r < p.out_rows) {
              const float g = __uint_as_float(v[cc]);
              if (S == 1)
                static_cast<__nv_bfloat16*>(p.out)[r * p.n_out + col] = __float2bfloat16_rn(g);
              else
                p.partial[(static_cast<long long>(s) * p.out_rows + r) * p.n_out + col] = g;
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
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// act[r, i] = SiLU(sum_s G_s[r, i]) * sum_s U_s[r, i] for r < offsets[E_r],
// splits added in order s = 0..S-1.  No-op when the GEMM chose S == 1.
__global__ void __launch_bounds__(256) split_swiglu_kernel(const float* __restrict__ partial,
                                                           const int32_t* __restrict__ split_word,
                                                           const int32_t* __restrict__ offsets,
                                                           int E_r, int I, long long out_rows,
                                                           __nv_bfloat16* __restrict__ act) {
  pdl_wait_and_trigger();
  const int S = *split_word;
  if (S <= 1) return;
  const long long n = min(static_cast<long long>(offsets[E_r]), out_rows);
  const int nq = I / 4;
  const long long total = n * nq;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / nq;
    const int c = static_cast<int>(i - r * nq) * 4;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    for (int s = 0; s < S; ++s) {
      const float* prow = partial + (static_cast<long long>(s) * out_rows + r) * 2 * I;
      const float4 a = __ldcg(reinterpret_cast<const float4*>(prow + c));
      const float4 b = __ldcg(reinterpret_cast<const float4*>(prow + I + c));
      g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
      u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
    }
    uint2 o;
    o.x = pack_bf16x2(silu_f(g.x) * u.x, silu_f(g.y) * u.y);
    o.y = pack_bf16x2(silu_f(g.z) * u.z, silu_f(g.w) * u.w);
    *reinterpret_cast<uint2*>(act + r * I + c) = o;
  }
}

// y[r, c] = sum_s Y_s[r, c] (split order) rounded to bf16, for r < offsets[E_r].
__global__ void __launch_bounds__(256) split_sum_kernel(const float* __restrict__ partial,
                                                        const int32_t* __restrict__ split_word,
                                                        const int32_t* __restrict__ offsets,
                                                        int E_r, int N, long long out_rows,
                                                        __nv_bfloat16* __restrict__ y) {
  pdl_wait_and_trigger();
  const int S = *split_word;
  if (S <= 1) return;
  const long long n = min(static_cast<long long>(offsets[E_r]), out_rows);
  const int nq = N / 4;
  const long long total = n * nq;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / nq;
    const int c = static_cast<int>(i - r * nq) * 4;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
      const float4 b =
          __ldcg(reinterpret_cast<const float4*>(partial + (static_cast<long long>(s) * out_rows + r) * N + c));
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    uint2 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    *reinterpret_cast<uint2*>(y + r * N + c) = o;
  }
}

template <bool GATE_UP, int STAGES, int CHUNK, int KSUB>
cudaError_t run_decode(const DecodeGemmArgs& a, cudaStream_t s) {
  using C = DCfg<GATE_UP, STAGES, CHUNK, KSUB>;
  CUtensorMap tw, tx, tx64;
  if (!make_tmap_bf16(&tw, a.w, a.w_rows, a.K, GATE_UP ? kGU : kM)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tx, a.x, a.x_rows, a.K, kTokBox)) return cudaErrorInvalidValue;
  if (!make_tmap_bf16(&tx64, a.x, a.x_rows, a.K, 64))
    return cudaErrorInvalidValue;
  DParams p;
  p.offsets = a.offsets;
  p.n_groups = a.n_groups;
  p.K = a.K;
  p.m_tiles = a.n_out / (GATE_UP ? kGU : kM);
  p.w_group_rows = a.w_group_rows;
  p.w_up_offset = GATE_UP ? a.n_out : 0;
  p.n_out = a.n_out;
  p.out = a.out;
  p.partial = a.partial;
  p.split_word = a.split_word;
  p.out_rows = a.out_rows;
  p.max_split = a.max_split;
  p.status = a.status;
  p.debug_flags = a.debug_flags;
  p.item_bytes = static_cast<float>(kM) * a.K * 2.f;
  p.total_scale = 1.f / 6200.f;  // ~6.2 TB/s sustained weight streaming
  auto kern = decode_gemm_kernel<GATE_UP, STAGES, CHUNK, KSUB>;
  static bool attr_done[64] = {false};
  cudaError_t e = set_smem_once(kern, static_cast<int>(C::kSmemBytes), attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(a.sm_count), dim3(kThreads), C::kSmemBytes, s, tw, tx, tx64, p);
}

}  // namespace

bool decode_gemm_supports(int n_out, bool gate_up) {
  return n_out % (gate_up ? kGU : kM) == 0;
}

cudaError_t launch_decode_gemm(const DecodeGemmArgs& a, cudaStream_t s) {
  if (a.x_rows <= 0) return cudaSuccess;
  if (a.gate_up) {
    cudaError_t e;
    if (a.chunk > 64)
      e = run_decode<true, 6, 128, 1>(a, s);
    else if (a.K % 128 == 0)
      e = run_decode<true, 4, 64, 2>(a, s);
    else
      e = run_decode<true, 8, 64, 1>(a, s);
    if (e != cudaSuccess || a.max_split <= 1) return e;
    return launch_pdl(split_swiglu_kernel, dim3(a.sm_count * 4), dim3(256), 0, s,
                      static_cast<const float*>(a.partial),
                      static_cast<const int32_t*>(a.split_word), a.offsets, a.n_groups, a.n_out,
                      a.out_rows, static_cast<__nv_bfloat16*>(a.out));
  }
  cudaError_t e;
  if (a.chunk > 64)
    e = run_decode<false, 4, 256, 1>(a, s);
  else if (a.K % 128 == 0)
    e = run_decode<false, 4, 64, 2>(a, s);
  else
    e = run_decode<false, 8, 64, 1>(a, s);
  if (e != cudaSuccess || a.max_split <= 1) return e;
  return launch_pdl(split_sum_kernel, dim3(a.sm_count * 4), dim3(256), 0, s,
                    static_cast<const float*>(a.partial), static_cast<const int32_t*>(a.split_word),
                    a.offsets, a.n_groups, a.n_out, a.out_rows,
                    static_cast<__nv_bfloat16*>(a.out));
}

}  // namespace moe
