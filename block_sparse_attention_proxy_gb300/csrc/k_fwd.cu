// Block-sparse attention forward, KV-major.
//
// The Flash-MSA summary (socker-news.uzaya.net, 要約) runs sparse attention
// through FlashAttention with MoBA's varlen trick: the queries that chose a
// KV block are gathered and attend to that block as one varlen problem.  Here
// one CTA owns one (KV group g, KV block b): K_b and V_b are staged once by
// TMA, then tiles of 128 rows = 128/G tokens x G heads are processed:
//   * first the block's own queries (the diagonal slot, causal inside the block),
//   * then the gathered queries from the regroup CSR (full block, no mask).
// Per tile: S = Q K^T on tcgen05 into TMEM, exact softmax over the block's 128
// keys (one TMEM lane = one row).  P goes back into the same TMEM columns as
// two bf16 operands, hi = bf16(P) and lo = bf16(P - hi) (16 hi and 16 lo
// columns in place of each 32 score columns, so no unread score is
// overwritten), and O = P_hi V + P_lo V reads P straight from TMEM; O keeps
// ~16 mantissa bits of P, which the backward's D = rowsum(dO * O) needs.  The
// normalised partial O_slot is written per (token, head, slot) as 16-bit fixed
// point relative to the row's max |O_slot| (int16 row + fp32 scale, beside
// lse_slot); the merge kernel combines the slots by log-sum-exp.
//
// Roles (384 threads): two softmax warpgroups (warps 0-3 and 4-7) take
// alternate tiles through two S/O accumulator pairs, so one warpgroup's
// softmax overlaps the other's P V product and O stores; warp 8 is the TMA
// producer (regroup entries read one tile ahead, four Q stages); warp 9 issues
// the MMAs; warps 10-11 only complete the third warpgroup, so that register
// budgets can be set per warpgroup (setmaxnreg): 2 x 128 x 200 for the softmax
// warps, 128 x 104 for the producer and MMA warps, 64512 = 384 x 168 in all (at
// 320 threads every warp was capped at 168 and the softmax warps spilled).
#include <cfloat>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kFwdThreads = 384;
constexpr uint32_t kFwdRegsSoftmax = 200, kFwdRegsCtl = 104;
constexpr int kFwdQStages = 4;
// Per softmax warp: a 32-row x 64-column int16 staging tile (128B-swizzled
// rows) and the 32 partial-row indices (-1: no row), used to turn
// row-per-thread O values into row-contiguous 128-byte segments, four rows
// per warp store.
constexpr int kFwdStageWarp = 4096 + 128;
constexpr float kLog2e = 1.4426950408889634f;

struct FwdArgs {
  const int32_t* cu;
  const int32_t* cu_blocks;
  const int32_t* row_ptr;
  const uint32_t* ent;
  int ndoc, T, hq, hkv, K, nb_bound;
  float scale;
  int16_t* o_part;  // [tokens of the query chunk (token - t0)][hq][K][D] int16
  float2* o_meta;   // [..][hq][K] {lse_slot, dequantisation scale}
  unsigned* status;
  int chunk;        // query chunk (qchunk_of)
  int qcb;          // KV blocks per query chunk
};

// Maximum of 32 scores held as raw fp32 bits (16 three-input max instructions).
__device__ __forceinline__ float max32_bits(const uint32_t (&r)[32]) {
  float m[11];
#pragma unroll
  for (int i = 0; i < 10; ++i)
    m[i] = fmax3(__uint_as_float(r[3 * i]), __uint_as_float(r[3 * i + 1]),
                 __uint_as_float(r[3 * i + 2]));
  m[10] = fmaxf(__uint_as_float(r[30]), __uint_as_float(r[31]));
  const float x = fmax3(m[0], m[1], m[2]), y = fmax3(m[3], m[4], m[5]);
  const float z = fmax3(m[6], m[7], m[8]);
  return fmax3(fmax3(x, y, z), m[9], m[10]);
}

template <int D, int G>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_fwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  constexpr int TPT = 128 / G;         // tokens per tile
  constexpr int TPL = (TPT + 31) / 32; // tokens per producer lane
  constexpr int NCH = D / 64;          // 64-column chunks of a head row
  constexpr int NQ = kFwdQStages;
  constexpr int kTile = 128 * D * 2;   // bytes of a 128-row, D-column bf16 tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + kTile;
  uint8_t* sQ = sV + kTile;  // [NQ]
  uint8_t* sOst = sQ + NQ * kTile;  // [8 warps] O staging
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOst + 8 * kFwdStageWarp);
  // [0] kv_full | [1, 1+NQ) q_full | [1+NQ, 1+2NQ) q_empty | then per accumulator
  // pair b in {0,1}: s_full, p_full, o_full, o_empty
  const int B_KV = 0, B_QF = 1, B_QE = 1 + NQ, B_ACC = 1 + 2 * NQ;
  auto b_sfull = [&](int b) { return B_ACC + 4 * b; };
  auto b_pfull = [&](int b) { return B_ACC + 4 * b + 1; };
  auto b_ofull = [&](int b) { return B_ACC + 4 * b + 2; };
  auto b_oempty = [&](int b) { return B_ACC + 4 * b + 3; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + B_ACC + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item ----
  if (!a.cu_blocks[a.ndoc + 1]) return;  // malformed cu_seqlens (flagged by k_meta)
  const int nbt = min(a.cu_blocks[a.ndoc], a.nb_bound);
  const int g = blockIdx.x % a.hkv;
  const int gb = (int)(blockIdx.x / a.hkv);
  if (gb >= nbt) return;
  const int d = doc_of_block(a.cu_blocks, a.ndoc, gb);
  const int j = gb - a.cu_blocks[d];
  const int dstart = a.cu[d];
  const int L = a.cu[d + 1] - dstart;
  const int kstart = dstart + j * kBlock;
  const int nkeys = min(kBlock, L - j * kBlock);
  // this launch's query chunk: the block's own queries if the block is in it,
  // and the part of its token-sorted list that falls in [t0, t1)
  const QChunk qc = qchunk_of(a.cu, a.cu_blocks, a.ndoc, a.T, nbt, a.chunk, a.qcb);
  int lbeg = a.row_ptr[g * a.nb_bound + gb];
  int lend = a.row_ptr[g * a.nb_bound + gb + 1];
  if (a.chunk >= 0) {
    lbeg = lower_bound_token(a.ent, lbeg, lend, qc.t0);
    lend = lower_bound_token(a.ent, lbeg, lend, qc.t1);
  }
  const int lcnt = lend - lbeg;
  const bool own = gb >= qc.b0 && gb < qc.b1;
  const int ndiag = own ? (nkeys + TPT - 1) / TPT : 0;
  const int ntiles = ndiag + (lcnt + TPT - 1) / TPT;
  if (ntiles == 0) return;
  const int slot_diag = min(j, a.K - 1);
  const int t0 = qc.t0;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_KV), 1);
    for (int s = 0; s < NQ; ++s) {
      mbar_init(bar(B_QF + s), 1);
      mbar_init(bar(B_QE + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(b_sfull(b)), 1);
      mbar_init(bar(b_pfull(b)), 4);
      mbar_init(bar(b_ofull(b)), 1);
      mbar_init(bar(b_oempty(b)), 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tslot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(tslot);
  // TMEM: S/P of pair b at columns [128 b, 128 b + 128), O of pair b at 256 + D b

  // token and slot of row-group i of tile n (T: out of range -> TMA zero fill)
  auto tile_token = [&](int n, int i, int& t, int& slot) -> bool {
    if (n < ndiag) {
      const int qi = n * TPT + i;
      t = kstart + qi;
      slot = slot_diag;
      return qi < nkeys && t < a.T;
    }
    const int m = (n - ndiag) * TPT + i;
    if (m >= lcnt) {
      t = a.T;
      slot = 0;
      return false;
    }
    const uint32_t e = __ldg(a.ent + lbeg + m);
    t = (int)(e >> 4);
    slot = (int)(e & 15u);
    return t < a.T;
  };

  if (warp >= 8) {
    setmaxnreg_dec<kFwdRegsCtl>();
    if (warp == 8) {
      // ------------------------------ TMA producer ------------------------------
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_KV), 2 * kTile);
  #pragma unroll
        for (int c = 0; c < NCH; ++c) {
          tma_load_3d(smem_u32(sK + c * 16384), &tm_k, bar(B_KV), 64 * c, g, kstart);
          tma_load_3d(smem_u32(sV + c * 16384), &tm_v, bar(B_KV), 64 * c, g, kstart);
        }
      }
      int tok[TPL];
      auto load_tokens = [&](int n) {
  #pragma unroll
        for (int u = 0; u < TPL; ++u) {
          const int i = lane + 32 * u;
          int t = a.T, slot;
          if (i < TPT && !tile_token(n, i, t, slot)) t = a.T;
          tok[u] = t;
        }
      };
      if (ntiles > 0) load_tokens(0);
      for (int n = 0; n < ntiles; ++n) {
        const int s = n % NQ;
        if (n >= NQ && !wait_bar_warp(bar(B_QE + s), ((n / NQ) & 1) ^ 1, abort_flag, a.status,
                                      wait_site(kKerFwd, B_QE + s, n)))
          break;
        int cur[TPL];
  #pragma unroll
        for (int u = 0; u < TPL; ++u) cur[u] = tok[u];
        if (n + 1 < ntiles) load_tokens(n + 1);
        if (lane == 0) mbar_arrive_expect_tx(bar(B_QF + s), kTile);
        __syncwarp();
        const uint32_t qb = smem_u32(sQ + s * kTile);
  #pragma unroll
        for (int u = 0; u < TPL; ++u) {
          const int i = lane + 32 * u;
          if (i < TPT) {
  #pragma unroll
            for (int c = 0; c < NCH; ++c)
              tma_load_3d(qb + c * 16384 + i * G * 128, &tm_q, bar(B_QF + s), 64 * c, g * G, cur[u]);
          }
        }
      }
    } else if (warp == 9) {
      // ------------------------------ MMA issuer ---------------------------------
      if (lane == 0) {
        constexpr uint32_t idS = make_idesc_bf16(128, 128, false, false);
        constexpr uint32_t idO = make_idesc_bf16(128, D, false, true);
        bool ok = wait_bar(bar(B_KV), 0, abort_flag, a.status, wait_site(kKerFwd, B_KV, 0));
        const uint32_t k0 = smem_u32(sK), v0 = smem_u32(sV);
        auto issue_s = [&](int n) -> bool {
          const int s = n % NQ, b = n & 1;
          if (!wait_bar(bar(B_QF + s), (n / NQ) & 1, abort_flag, a.status,
                        wait_site(kKerFwd, B_QF + s, n)))
            return false;
          // S(n) overwrites the P of tile n-2: wait until that P V has completed
          if (n >= 2 && !wait_bar(bar(b_ofull(b)), ((n - 2) >> 1) & 1, abort_flag, a.status,
                                  wait_site(kKerFwd, b_ofull(b), n)))
            return false;
          tc_fence_after();
          const uint32_t q0 = smem_u32(sQ + s * kTile);
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_bf16(tbase + 128 * b, make_sdesc(q0 + off, 16, 1024, kLayoutSW128),
                      make_sdesc(k0 + off, 16, 1024, kLayoutSW128), idS, kk > 0);
          }
          umma_commit(bar(b_sfull(b)));
          umma_commit(bar(B_QE + s));
          return true;
        };
        if (ok && ntiles > 0) ok = issue_s(0);
        for (int n = 1; ok && n <= ntiles; ++n) {
          // P V for tile n-1, then S for tile n
          const int m = n - 1, b = m & 1;
          if (!wait_bar(bar(b_pfull(b)), (m >> 1) & 1, abort_flag, a.status,
                        wait_site(kKerFwd, b_pfull(b), m)))
            break;
          if (m >= 2 && !wait_bar(bar(b_oempty(b)), ((m >> 1) & 1) ^ 1, abort_flag, a.status,
                                  wait_site(kKerFwd, b_oempty(b), m)))
            break;
          tc_fence_after();
          const uint32_t pa = tbase + 128 * b;
  #pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // keys 16kk..16kk+15: hi at column 32(kk/2) + 8(kk%2), lo 16 columns further
            const uint32_t ph = pa + 32 * (kk >> 1) + 8 * (kk & 1);
            const uint64_t bd = make_sdesc(v0 + kk * 2048, 16384, 1024, kLayoutSW128);
            umma_bf16_ts(tbase + 256 + b * D, ph, bd, idO, kk > 0);
            umma_bf16_ts(tbase + 256 + b * D, ph + 16, bd, idO, 1u);
          }
          umma_commit(bar(b_ofull(b)));
          if (n < ntiles && !issue_s(n)) break;
        }
      }
    }
  } else {
    setmaxnreg_inc<kFwdRegsSoftmax>();
    // ------------------------------ softmax / epilogue --------------------------
    // Warpgroup e takes tiles n = e, e + 2, ... through accumulator pair e.
    // Abort-safe: a failed wait marks the warp dead; it keeps walking its tiles
    // and arriving on its barriers without touching TMEM.
    const int e = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int ti = row / G, hl = row % G;
    const float sl2 = a.scale * kLog2e;
    bool dead = false;
    // the row's list entry (token, slot) is read one tile ahead: its global
    // load then overlaps the wait for the scores instead of stalling the O store
    int t_nx = a.T, slot_nx = 0;
    bool valid_nx = e < ntiles && tile_token(e, ti, t_nx, slot_nx);
    for (int n = e; n < ntiles; n += 2) {
      const int b = e, ph = (n >> 1) & 1;
      const int t = t_nx, slot = slot_nx;
      const bool valid = valid_nx;
      if (n + 2 < ntiles) valid_nx = tile_token(n + 2, ti, t_nx, slot_nx);
      const bool diag = n < ndiag;
      const int qpos = n * TPT + ti;  // position inside the block (diagonal tiles)
      dead = dead || !wait_bar_warp(bar(b_sfull(b)), ph, abort_flag, a.status,
                                    wait_site(kKerFwd, b_sfull(b), n));
      tc_fence_after();
      const uint32_t ts = tbase + lane_off + 128 * b;
      float mx = -FLT_MAX, l = 0.f;
      if (!dead) {
        // row maximum: 64 columns per TMEM round trip, three-input max tree
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t va[32], vb[32];
          tmem_ld32x2(ts + c2 * 64, ts + c2 * 64 + 32, va, vb);
          if (diag) {
            const uint32_t neg = __float_as_uint(-FLT_MAX);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (c2 * 64 + i > qpos) va[i] = neg;
              if (c2 * 64 + 32 + i > qpos) vb[i] = neg;
            }
          }
          mx = fmax3(mx, max32_bits(va), max32_bits(vb));
        }
        const float mb = mx * sl2;
        float l4[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums: no serial add chain
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tmem_ld32f(ts + c * 32, v);
          uint32_t w[32];  // 16 hi words then 16 lo words (keys 32c .. 32c+31)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int k0 = c * 32 + 2 * i;
            float p0 = ex2_approx(fmaf(v[2 * i], sl2, -mb));
            float p1 = ex2_approx(fmaf(v[2 * i + 1], sl2, -mb));
            if (diag) {
              p0 = k0 <= qpos ? p0 : 0.f;
              p1 = k0 + 1 <= qpos ? p1 : 0.f;
            }
            l4[i & 3] += p0 + p1;
            const uint32_t hi = pack_bf16(p0, p1);
            w[i] = hi;
            w[16 + i] = pack_bf16(p0 - bf16_lo(hi), p1 - bf16_hi(hi));
          }
          tmem_st32(ts + c * 32, w);
        }
        l = (l4[0] + l4[1]) + (l4[2] + l4[3]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(b_pfull(b)));
      dead = dead || !wait_bar_warp(bar(b_ofull(b)), ph, abort_flag, a.status,
                                    wait_site(kKerFwd, b_ofull(b), n));
      tc_fence_after();
      if (!dead) {
        // O row (this thread's): a first pass over TMEM finds max |O|, a second
        // writes it as 16-bit fixed point, 64 columns per TMEM round trip:
        // registers -> swizzled staging tile -> each warp store writes 4 rows
        // x 128 contiguous bytes.
        const uint32_t to = tbase + lane_off + 256 + b * D;
        uint32_t mbits = 0;
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          uint32_t va[32], vb[32];
          tmem_ld32x2(to + c * 64, to + c * 64 + 32, va, vb);
#pragma unroll
          for (int i = 0; i < 32; ++i) mbits = max(mbits, max(abs_bits(va[i]), abs_bits(vb[i])));
        }
        const float mo = __uint_as_float(mbits);
        const float qf = q16_factor(mo);
        uint8_t* stg = sOst + warp * kFwdStageWarp;
        // partial rows of one query chunk: < 262144 tokens x 255 heads x 16 slots < 2^31
        int32_t* rowi = reinterpret_cast<int32_t*>(stg + 4096);
        const size_t prow = ((size_t)(t - t0) * a.hq + g * G + hl) * a.K + slot;
        rowi[lane] = valid ? (int32_t)prow : -1;
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          uint32_t va[32], vb[32];
          tmem_ld32x2(to + c * 64, to + c * 64 + 32, va, vb);
          uint32_t w[32];  // columns 64c .. 64c+63 as int16 pairs
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = pack_q16x2(__uint_as_float(va[2 * i]) * qf, __uint_as_float(va[2 * i + 1]) * qf);
            w[16 + i] =
                pack_q16x2(__uint_as_float(vb[2 * i]) * qf, __uint_as_float(vb[2 * i + 1]) * qf);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          __syncwarp();
          const int ch = lane & 7;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = (lane >> 3) + 4 * i;
            const uint4 x = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((ch ^ (rr & 7)) << 4));
            const int32_t ri = rowi[rr];
            if (ri >= 0)
              *reinterpret_cast<uint4*>(a.o_part + (size_t)ri * D + c * 64 + ch * 8) = x;
          }
          __syncwarp();
        }
        // O_slot = O / l, so the row's factor is max|O| / (32767 l)
        if (valid) a.o_meta[prow] = make_float2(mx * a.scale + __logf(l), mo / (kQ16 * l));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(b_oempty(b)));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace
}  // namespace msa

namespace msa {
namespace {

template <int D, int G>
cudaError_t launch_fwd_t(const Shape& s, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const FwdArgs& a, cudaStream_t st) {
  const size_t smem = 1024 + (2 + kFwdQStages) * (128 * D * 2) + 8 * kFwdStageWarp + 256;
  static_assert(1024 + (2 + kFwdQStages) * (128 * 128 * 2) + 8 * kFwdStageWarp + 256 <= 232448,
                "shared memory budget");
  // The warpgroups' register budgets are drawn from the registers the block
  // is launched with; a larger sum would leave setmaxnreg.inc waiting.
  constexpr int kBudget = 2 * 128 * kFwdRegsSoftmax + 128 * kFwdRegsCtl;
  static_assert(kBudget <= 65536, "register budgets exceed the register file");
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, k_fwd<D, G>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kFwdThreads < kBudget) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(k_fwd<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_fwd<D, G><<<s.nb_bound * s.hkv, kFwdThreads, smem, st>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_fwd_d(const Shape& s, const CUtensorMap& mq, const CUtensorMap& mk,
                         const CUtensorMap& mv, const FwdArgs& a, cudaStream_t st) {
  switch (s.G) {
    case 1: return launch_fwd_t<D, 1>(s, mq, mk, mv, a, st);
    case 2: return launch_fwd_t<D, 2>(s, mq, mk, mv, a, st);
    case 4: return launch_fwd_t<D, 4>(s, mq, mk, mv, a, st);
    default: return launch_fwd_t<D, 8>(s, mq, mk, mv, a, st);
  }
}

}  // namespace

cudaError_t launch_fwd(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                       const int32_t* row_ptr, const uint32_t* ent, const uint16_t* q,
                       const uint16_t* k, const uint16_t* v, int16_t* o_part, float2* o_meta,
                       int chunk, unsigned* status, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  cudaError_t e;
  if ((e = make_tmap_3d(&mq, q, s.d, s.hq, s.T, 64, s.G, 1, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&mk, k, s.d, s.hkv, s.T, 64, 1, 128, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&mv, v, s.d, s.hkv, s.T, 64, 1, 128, 128)) != cudaSuccess) return e;
  FwdArgs a{cu_seqlens, cu_blocks, row_ptr, ent,   s.ndoc, s.T,   s.hq,
            s.hkv,      s.K,       s.nb_bound, s.softmax_scale, o_part, o_meta,   status,
            chunk,      s.qc_blocks};
  return s.d == 128 ? launch_fwd_d<128>(s, mq, mk, mv, a, st)
                    : launch_fwd_d<64>(s, mq, mk, mv, a, st);
}

}  // namespace msa
