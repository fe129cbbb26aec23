// Block-sparse attention backward with the fused proxy-KL gradient, KV-major.
//
// The pages fuse the backward passes of the proxy and of the main attention
// ("... 'Flash-MSA' ...", ai-minor.com, "Why Does This Matter?", fused
// backward).  One CTA owns one (KV group g, KV block b), as in the forward:
// K_b, V_b are staged once; tiles of 64 rows (64/G tokens x G heads) run the
// block's own queries (causal) and then the gathered queries.  The transposed
// form keeps one key per TMEM lane:
//   S^T  = K Q^T       dP^T = V dO^T                     (tcgen05, TMEM)
//   P^T  = exp(scale S^T - LSE_row),  dS^T = scale P^T (dP^T - D_row)
//   dV  += P^T dO      dK  += dS^T Q                     (TMEM, whole block)
//   dQ^T = K^T dS^T                                      (TMEM, per tile)
// dK and dV stay in TMEM for all tiles of the block and are written once; dQ
// is written per (token, head, slot) in fp32 and summed by the reduce kernel.
// dS enters the dK and dQ products as two bf16 operands, hi = bf16(dS) and
// lo = bf16(dS - hi), so the products keep about 16 mantissa bits of dS.
// Fused proxy part: every (token, slot) of the block's list carries
//   g_b = kl_weight * proxy_scale * (exp(S_b - plse) - m_b),
// and the epilogue thread that owns key a_b adds g_b q_p[t] to its register
// copy of dk_p[a_b] (tokens in list order, so the sum is deterministic); the
// block's dk_p rows are written once at the end.
//
// Per-row metadata comes from k_bwd_prep, which lays one record per list
// entry (token, slot, argmax, g_b, and LSE and D of the token's G heads)
// contiguously in the list's order, so a tile's metadata is one bulk copy.
//
// Roles (320 threads): warps 0-7 epilogue (two warpgroups, each half of a
// tile's rows), warp 8 TMA producer, warp 9 MMA issuer.  Stages of {Q, dO, q_p rows, records} are multi-buffered; the next
// tile's S^T/dP^T products run while the epilogue stores the previous dQ.
#include <cfloat>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kBwdThreads = 320;
constexpr int kRT = 64;  // rows per tile
constexpr float kLog2eB = 1.4426950408889634f;

template <int D, int G, int DP>
struct BwdCfg {
  static constexpr int TPT = kRT / G;             // tokens per tile
  static constexpr int TPL = (TPT + 31) / 32;     // tokens per producer lane
  static constexpr int kKV = 128 * D * 2;         // K or V tile
  static constexpr int kQT = kRT * D * 2;         // Q or dO tile (64 rows)
  static constexpr int kQChunk = kRT * 128;       // one 64-column chunk of a Q/dO tile
  static constexpr int kQpRow = 128;              // q_p rows land at a 128-byte stride
  static constexpr int kRec = bwd_rec_bytes(G);
  static constexpr int kStage = 2 * kQT + TPT * kQpRow + TPT * kRec;
  static constexpr int kStageAl = (kStage + 1023) / 1024 * 1024;
  static constexpr int kFixed = 2 * kKV + 3 * 16384;  // K, V, P^T, dS^T hi, dS^T lo
  static constexpr int kBars = 256;
  static constexpr int kNS = (1024 + kFixed + 3 * kStageAl + kBars <= 232448) ? 3 : 2;
  static constexpr int kSmem = 1024 + kFixed + kNS * kStageAl + kBars;
};

struct BwdArgs {
  const int32_t* cu;
  const int32_t* cu_blocks;
  const int32_t* row_ptr;
  const uint32_t* ent;
  const uint8_t* rec;  // list-entry records (k_bwd_prep)
  const float* lse;
  const float* dsum;
  const float* mass;
  const float* sel_score;
  const uint8_t* sel_arg;
  const float* plse;
  int ndoc, T, hq, hkv, K, nb_bound;
  float scale, proxy_scale, kl_weight;
  float* dq_part;
  float* dk;
  float* dv;
  float* dk_p;
  unsigned* status;
};

// Work item of CTA `x`: KV group g, global block gb, the block's token range
// and its list (diagonal tokens first, then the gathered entries).
struct Item {
  int g, gb, j, kstart, nkeys, lbeg, lcnt, ndiag, ntiles, slot_diag;
  long long ext;  // index of the item's first record
};

__device__ __forceinline__ bool item_of(int x, int TPT, const BwdArgs& a, Item& it) {
  if (!a.cu_blocks[a.ndoc + 1]) return false;  // malformed cu_seqlens (flagged by k_meta)
  const int nbt = min(a.cu_blocks[a.ndoc], a.nb_bound);
  it.g = x % a.hkv;
  it.gb = x / a.hkv;
  if (it.gb >= nbt) return false;
  const int d = doc_of_block(a.cu_blocks, a.ndoc, it.gb);
  it.j = it.gb - a.cu_blocks[d];
  const int dstart = a.cu[d];
  const int L = a.cu[d + 1] - dstart;
  it.kstart = dstart + it.j * kBlock;
  it.nkeys = min(kBlock, L - it.j * kBlock);
  it.lbeg = a.row_ptr[it.g * a.nb_bound + it.gb];
  it.lcnt = a.row_ptr[it.g * a.nb_bound + it.gb + 1] - it.lbeg;
  it.ndiag = (it.nkeys + TPT - 1) / TPT;
  it.ntiles = it.ndiag + (it.lcnt + TPT - 1) / TPT;
  it.slot_diag = min(it.j, a.K - 1);
  // Records of group g follow those of groups < g (their lists plus T diagonal
  // entries each); inside the group, block gb's diagonal entries are preceded
  // by kstart diagonal entries of earlier blocks.
  it.ext = (long long)it.lbeg + (long long)it.g * a.T + it.kstart;
  return true;
}

// First list entry and entry count of tile n.
__device__ __forceinline__ void tile_span(const Item& it, int n, int TPT, int& x0, int& cnt) {
  if (n < it.ndiag) {
    x0 = n * TPT;
    cnt = min(TPT, it.nkeys - x0);
  } else {
    const int m = (n - it.ndiag) * TPT;
    x0 = it.nkeys + m;
    cnt = min(TPT, it.lcnt - m);
  }
}

// One record per list entry of every work item, in list order:
//   int {t, slot, arg, g_b bits} then G x float {LSE, D}, padded to 16 bytes.
// Entries with an out-of-range token are written with t = T (the kernel then
// treats them as padding).
template <int G>
__global__ void __launch_bounds__(128) k_bwd_prep(const BwdArgs a) {
  constexpr int kRec = bwd_rec_bytes(G);
  Item it;
  if (!item_of(blockIdx.x, kRT / G, a, it)) return;
  const int n_ext = it.nkeys + it.lcnt;
  const float gscale = a.kl_weight * a.proxy_scale;
  for (int x = threadIdx.x; x < n_ext; x += blockDim.x) {
    int t, slot;
    if (x < it.nkeys) {
      t = it.kstart + x;
      slot = it.slot_diag;
    } else {
      const uint32_t e = __ldg(a.ent + it.lbeg + (x - it.nkeys));
      t = (int)(e >> 4);
      slot = (int)(e & 15u);
    }
    int4 hdr = make_int4(a.T, 0, 0, 0);
    float2 rows[G];
#pragma unroll
    for (int h = 0; h < G; ++h) rows[h] = make_float2(__int_as_float(0x7f800000), 0.f);
    if (t >= 0 && t < a.T) {
      const size_t e = ((size_t)t * a.hkv + it.g) * a.K + slot;
      const float p = __expf(__ldg(a.sel_score + e) - __ldg(a.plse + (size_t)t * a.hkv + it.g));
      const float gs = gscale * (p - __ldg(a.mass + e));
      hdr = make_int4(t, slot, __ldg(a.sel_arg + e) & (kBlock - 1), __float_as_int(gs));
      const size_t r0 = (size_t)t * a.hq + it.g * G;
#pragma unroll
      for (int h = 0; h < G; ++h) rows[h] = make_float2(__ldg(a.lse + r0 + h), __ldg(a.dsum + r0 + h));
    }
    uint8_t* dst = const_cast<uint8_t*>(a.rec) + (size_t)(it.ext + x) * kRec;
    *reinterpret_cast<int4*>(dst) = hdr;
#pragma unroll
    for (int h = 0; h < G; h += 2) {
      const float2 r1 = (h + 1 < G) ? rows[h + 1] : make_float2(0.f, 0.f);
      *reinterpret_cast<float4*>(dst + 16 + 8 * h) = make_float4(rows[h].x, rows[h].y, r1.x, r1.y);
    }
  }
}

template <int D, int G, int DP>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_bwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
          const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
          const __grid_constant__ CUtensorMap tm_qp, const BwdArgs a) {
  using C = BwdCfg<D, G, DP>;
  constexpr int TPT = C::TPT, TPL = C::TPL, NS = C::kNS, NCH = D / 64;
  constexpr int kQT = C::kQT, kQChunk = C::kQChunk, kRec = C::kRec;
  constexpr uint32_t T_S = 0, T_DP = 64, T_DV = 128, T_DK = 128 + D, T_DQ = 128 + 2 * D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::kKV;
  uint8_t* sPs = sV + C::kKV;    // P^T  [128 keys][64 rows] bf16, 128B swizzle
  uint8_t* sdS = sPs + 16384;    // dS^T hi
  uint8_t* sdSl = sdS + 16384;   // dS^T lo; sPs..sdS double as the fp32 dQ stage
  uint8_t* sStage = sdSl + 16384;
  auto stQ = [&](int s) { return sStage + s * C::kStageAl; };
  auto stO = [&](int s) { return stQ(s) + kQT; };
  auto stP = [&](int s) { return stQ(s) + 2 * kQT; };           // q_p rows
  auto stR = [&](int s) { return stP(s) + TPT * C::kQpRow; };   // records
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + NS * C::kStageAl);
  const int B_FULL = 0, B_FREE = NS, B_SP = 2 * NS, B_DS = 2 * NS + 1, B_DQ = 2 * NS + 2,
            B_DQT = 2 * NS + 3, B_KV = 2 * NS + 4;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * NS + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Item it;
  if (!item_of(blockIdx.x, TPT, a, it)) return;
  const int g = it.g;
  const uint8_t* recg = a.rec + (size_t)it.ext * kRec;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_FREE + s), 8);
    }
    mbar_init(bar(B_SP), 1);
    mbar_init(bar(B_DS), 8);
    mbar_init(bar(B_DQ), 1);
    mbar_init(bar(B_DQT), 8);
    mbar_init(bar(B_KV), 1);
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

  if (warp == 8) {
    // ------------------------------ TMA producer --------------------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(B_KV), 2 * C::kKV);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d(smem_u32(sK + c * 16384), &tm_k, bar(B_KV), 64 * c, g, it.kstart);
        tma_load_3d(smem_u32(sV + c * 16384), &tm_v, bar(B_KV), 64 * c, g, it.kstart);
      }
    }
    // tokens of the next tile are read one tile ahead (records hold them)
    int tok[TPL];
    auto load_tokens = [&](int n) {
      int x0, cnt;
      tile_span(it, n, TPT, x0, cnt);
#pragma unroll
      for (int u = 0; u < TPL; ++u) {
        const int i = lane + 32 * u;
        tok[u] = (i < TPT && i < cnt)
                     ? __ldg(reinterpret_cast<const int*>(recg + (size_t)(x0 + i) * kRec))
                     : a.T;
      }
    };
    if (it.ntiles > 0) load_tokens(0);
    for (int n = 0; n < it.ntiles; ++n) {
      const int s = n % NS;
      if (n >= NS && !wait_bar_warp(bar(B_FREE + s), ((n / NS) & 1) ^ 1, abort_flag, a.status,
                                    wait_site(kKerBwd, B_FREE + s, n)))
        break;
      int cur[TPL];
#pragma unroll
      for (int u = 0; u < TPL; ++u) cur[u] = tok[u];
      if (n + 1 < it.ntiles) load_tokens(n + 1);
      int x0, cnt;
      tile_span(it, n, TPT, x0, cnt);
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_FULL + s), 2 * kQT + TPT * DP * 2 + TPT * kRec);
        bulk_load(smem_u32(stR(s)), recg + (size_t)x0 * kRec, TPT * kRec, bar(B_FULL + s));
      }
      __syncwarp();
      const uint32_t qb = smem_u32(stQ(s)), ob = smem_u32(stO(s)), pb = smem_u32(stP(s));
#pragma unroll
      for (int u = 0; u < TPL; ++u) {
        const int i = lane + 32 * u;
        if (i < TPT) {
          const int t = cur[u];
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            tma_load_3d(qb + c * kQChunk + i * G * 128, &tm_q, bar(B_FULL + s), 64 * c, g * G, t);
            tma_load_3d(ob + c * kQChunk + i * G * 128, &tm_do, bar(B_FULL + s), 64 * c, g * G, t);
          }
          tma_load_3d(pb + i * C::kQpRow, &tm_qp, bar(B_FULL + s), 0, g, t);
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------ MMA issuer ---------------------------------
    if (lane == 0) {
      constexpr uint32_t idST = make_idesc_bf16(128, kRT, false, false);
      constexpr uint32_t idDV = make_idesc_bf16(128, D, false, true);
      constexpr uint32_t idDQ = make_idesc_bf16(128, kRT, true, true);
      bool ok = wait_bar(bar(B_KV), 0, abort_flag, a.status, wait_site(kKerBwd, B_KV, 0));
      const uint32_t k0 = smem_u32(sK), v0 = smem_u32(sV);
      const uint32_t ps0 = smem_u32(sPs), ds0 = smem_u32(sdS), dl0 = smem_u32(sdSl);
      for (int n = 0; ok && n < it.ntiles; ++n) {
        const int s = n % NS;
        if (!wait_bar(bar(B_FULL + s), (n / NS) & 1, abort_flag, a.status,
                      wait_site(kKerBwd, B_FULL + s, n)))
          break;
        tc_fence_after();
        const uint32_t q0 = smem_u32(stQ(s)), o0 = smem_u32(stO(s));
        // S^T = K Q^T and dP^T = V dO^T   (M = 128 keys, N = 64 rows, K = D)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t kv_off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t q_off = (kk >> 2) * kQChunk + (kk & 3) * 32;
          umma_bf16(tbase + T_S, make_sdesc(k0 + kv_off, 16, 1024, kLayoutSW128),
                    make_sdesc(q0 + q_off, 16, 1024, kLayoutSW128), idST, kk > 0);
          umma_bf16(tbase + T_DP, make_sdesc(v0 + kv_off, 16, 1024, kLayoutSW128),
                    make_sdesc(o0 + q_off, 16, 1024, kLayoutSW128), idST, kk > 0);
        }
        umma_commit(bar(B_SP));
        if (!wait_bar(bar(B_DS), n & 1, abort_flag, a.status, wait_site(kKerBwd, B_DS, n))) break;
        if (n >= 1 && !wait_bar(bar(B_DQT), (n - 1) & 1, abort_flag, a.status,
                                wait_site(kKerBwd, B_DQT, n)))
          break;
        tc_fence_after();
        // dV += P^T dO, dK += (dS_hi + dS_lo)^T Q   (M = 128 keys, N = D, K = 64 rows)
#pragma unroll
        for (int kk = 0; kk < kRT / 16; ++kk) {
          const uint32_t acc = (n > 0 || kk > 0) ? 1u : 0u;
          const uint64_t bdo = make_sdesc(o0 + kk * 2048, kQChunk, 1024, kLayoutSW128);
          const uint64_t bq = make_sdesc(q0 + kk * 2048, kQChunk, 1024, kLayoutSW128);
          umma_bf16(tbase + T_DV, make_sdesc(ps0 + kk * 32, 16, 1024, kLayoutSW128), bdo, idDV,
                    acc);
          umma_bf16(tbase + T_DK, make_sdesc(ds0 + kk * 32, 16, 1024, kLayoutSW128), bq, idDV,
                    acc);
          umma_bf16(tbase + T_DK, make_sdesc(dl0 + kk * 32, 16, 1024, kLayoutSW128), bq, idDV, 1u);
        }
        // dQ^T = K^T (dS_hi + dS_lo)^T   (M = D (padded to 128), N = 64 rows, K = 128 keys)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ak = make_sdesc(k0 + kk * 2048, 16384, 1024, kLayoutSW128);
          umma_bf16(tbase + T_DQ, ak, make_sdesc(ds0 + kk * 2048, 16384, 1024, kLayoutSW128),
                    idDQ, kk > 0);
          umma_bf16(tbase + T_DQ, ak, make_sdesc(dl0 + kk * 2048, 16384, 1024, kLayoutSW128),
                    idDQ, 1u);
        }
        umma_commit(bar(B_DQ));
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------------
    // Two warpgroups: warpgroup e owns tile rows 32e..32e+31 (columns of S^T,
    // dP^T and dQ^T) for all 128 keys.  Abort-safe: a failed wait marks the
    // warp dead; it still walks every tile and every named barrier.
    const int e = warp >> 2;
    const int kk = (warp & 3) * 32 + lane;  // key (S^T/dP^T/dV/dK lanes) or d index (dQ^T lanes)
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale * kLog2eB;
    const bool unit_scale = a.scale == 1.f;
    float kp[DP];  // this warpgroup's share of the dk_p row of key kk
#pragma unroll
    for (int u = 0; u < DP; ++u) kp[u] = 0.f;
    bool dead = false;
    for (int n = 0; n < it.ntiles; ++n) {
      const int s = n % NS;
      int x0, cnt;
      tile_span(it, n, TPT, x0, cnt);
      const bool diag = n < it.ndiag;
      const bool masked = diag || cnt < TPT;
      const uint8_t* rec = stR(s);
      dead = dead || !wait_bar_warp(bar(B_FULL + s), (n / NS) & 1, abort_flag, a.status,
                                    wait_site(kKerBwd, B_FULL + s, n));
      dead = dead || !wait_bar_warp(bar(B_SP), n & 1, abort_flag, a.status,
                                    wait_site(kKerBwd, B_SP, n));
      tc_fence_after();
      if (!dead) {
#pragma unroll
        for (int q16 = 0; q16 < 2; ++q16) {
          const int r0 = 32 * e + 16 * q16;
          uint32_t sv[16], dv[16];
          tmem_ld16x2(tbase + lane_off + T_S + r0, tbase + lane_off + T_DP + r0, sv, dv);
          uint32_t pp[8], dh[8], dl[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float pv[2], hv[2], lv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int r = r0 + 2 * i + u;
              const int ti = r / G, hl = r % G;
              const float2 ld = *reinterpret_cast<const float2*>(rec + ti * kRec + 16 + 8 * hl);
              float p = ex2_approx(fmaf(__uint_as_float(sv[2 * i + u]), sl2, -ld.x * kLog2eB));
              float ds = p * (__uint_as_float(dv[2 * i + u]) - ld.y);
              if (!unit_scale) ds *= a.scale;
              if (masked) {
                const bool use = ti < cnt && (!diag || kk <= x0 + ti);
                p = use ? p : 0.f;
                ds = use ? ds : 0.f;
              }
              pv[u] = p;
              hv[u] = __bfloat162float(__float2bfloat16_rn(ds));
              lv[u] = ds - hv[u];
            }
            pp[i] = pack_bf16(pv[0], pv[1]);
            dh[i] = pack_bf16(hv[0], hv[1]);
            dl[i] = pack_bf16(lv[0], lv[1]);
          }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint32_t off = sw128_offset((uint32_t)kk, (uint32_t)(r0 / 8 + q));
            *reinterpret_cast<uint4*>(sPs + off) =
                make_uint4(pp[4 * q], pp[4 * q + 1], pp[4 * q + 2], pp[4 * q + 3]);
            *reinterpret_cast<uint4*>(sdS + off) =
                make_uint4(dh[4 * q], dh[4 * q + 1], dh[4 * q + 2], dh[4 * q + 3]);
            *reinterpret_cast<uint4*>(sdSl + off) =
                make_uint4(dl[4 * q], dl[4 * q + 1], dl[4 * q + 2], dl[4 * q + 3]);
          }
        }
        // fused proxy gradient: tokens (this warpgroup takes every other one)
        // whose block argmax is this thread's key
        for (int i = e; i < cnt; i += 2) {
          const int4 hd = *reinterpret_cast<const int4*>(rec + i * kRec);
          if (hd.z == kk && hd.x < a.T) {
            const float gs = __int_as_float(hd.w);
            const uint4* qrow = reinterpret_cast<const uint4*>(stP(s) + i * C::kQpRow);
#pragma unroll
            for (int u = 0; u < DP / 8; ++u) {
              const uint4 w = qrow[u];
              kp[8 * u + 0] = fmaf(gs, bf16_lo(w.x), kp[8 * u + 0]);
              kp[8 * u + 1] = fmaf(gs, bf16_hi(w.x), kp[8 * u + 1]);
              kp[8 * u + 2] = fmaf(gs, bf16_lo(w.y), kp[8 * u + 2]);
              kp[8 * u + 3] = fmaf(gs, bf16_hi(w.y), kp[8 * u + 3]);
              kp[8 * u + 4] = fmaf(gs, bf16_lo(w.z), kp[8 * u + 4]);
              kp[8 * u + 5] = fmaf(gs, bf16_hi(w.z), kp[8 * u + 5]);
              kp[8 * u + 6] = fmaf(gs, bf16_lo(w.w), kp[8 * u + 6]);
              kp[8 * u + 7] = fmaf(gs, bf16_hi(w.w), kp[8 * u + 7]);
            }
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DS));
      dead = dead || !wait_bar_warp(bar(B_DQ), n & 1, abort_flag, a.status,
                                    wait_site(kKerBwd, B_DQ, n));
      tc_fence_after();
      // dQ^T: lane kk = head-dim index; this warpgroup's 32 row columns go to the
      // fp32 stage [row][D] laid over sPs/sdS
      float* stage = reinterpret_cast<float*>(sPs);
      if (!dead) {
        uint32_t v0[16], v1[16];
        tmem_ld16x2(tbase + lane_off + T_DQ + 32 * e, tbase + lane_off + T_DQ + 32 * e + 16, v0,
                    v1);
        if (kk < D) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            stage[(32 * e + i) * D + kk] = __uint_as_float(v0[i]);
            stage[(32 * e + 16 + i) * D + kk] = __uint_as_float(v1[i]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DQT));  // the MMA may overwrite dQ^T now
      named_bar_sync(1 + e, 128);
      constexpr int TPR = D / 4;      // threads per row (16 bytes each)
      constexpr int RPI = 128 / TPR;  // rows per iteration
      if (!dead) {
        const int tid = (warp & 3) * 32 + lane;
#pragma unroll 4
        for (int itn = 0; itn < 32 / RPI; ++itn) {
          const int r = 32 * e + itn * RPI + tid / TPR, c = tid % TPR;
          const int ti = r / G;
          if (ti < cnt) {
            const int4 hd = *reinterpret_cast<const int4*>(rec + ti * kRec);
            if (hd.x < a.T) {
              float* dst = a.dq_part +
                           (((size_t)hd.x * a.hq + g * G + r % G) * a.K + hd.y) * (size_t)D + c * 4;
              *reinterpret_cast<float4*>(dst) =
                  *reinterpret_cast<const float4*>(stage + r * D + c * 4);
            }
          }
        }
      }
      named_bar_sync(1 + e, 128);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_FREE + s));
    }
    // dK, dV and dk_p rows of this block (lane = key), written once.  Warpgroup
    // 1 hands its dk_p partial over through shared memory; warpgroup 0 adds it
    // (a fixed order) and writes dk_p and dV, warpgroup 1 writes dK.  The TMEM
    // loads are warp-collective, so every lane executes them; only the stores
    // depend on the key being inside the document.
    float* kbuf = reinterpret_cast<float*>(sPs);  // [DP][128]
    named_bar_sync(3, 256);
    if (e == 1) {
#pragma unroll
      for (int u = 0; u < DP; ++u) kbuf[u * 128 + kk] = kp[u];
    }
    named_bar_sync(3, 256);
    tc_fence_after();
    if (!dead) {
      const bool keep = kk < it.nkeys;
      const size_t krow = (size_t)(it.kstart + (keep ? kk : 0)) * a.hkv + g;
      float* outr = (e == 0 ? a.dv : a.dk) + krow * D;
      const uint32_t tcol = e == 0 ? T_DV : T_DK;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32f(tbase + lane_off + tcol + c * 32, v);
        if (keep) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(outr + c * 32)[q] =
                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
      if (keep && e == 0) {
        float* pr = a.dk_p + krow * DP;
#pragma unroll
        for (int q = 0; q < DP / 4; ++q)
          reinterpret_cast<float4*>(pr)[q] =
              make_float4(kp[4 * q] + kbuf[(4 * q) * 128 + kk],
                          kp[4 * q + 1] + kbuf[(4 * q + 1) * 128 + kk],
                          kp[4 * q + 2] + kbuf[(4 * q + 2) * 128 + kk],
                          kp[4 * q + 3] + kbuf[(4 * q + 3) * 128 + kk]);
      }
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

template <int D, int G, int DP>
cudaError_t launch_bwd_t(const Shape& s, const CUtensorMap* m, const BwdArgs& a, cudaStream_t st) {
  using C = BwdCfg<D, G, DP>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  k_bwd_prep<G><<<s.nb_bound * s.hkv, 128, 0, st>>>(a);
  cudaError_t e = cudaFuncSetAttribute(k_bwd<D, G, DP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  k_bwd<D, G, DP><<<s.nb_bound * s.hkv, kBwdThreads, C::kSmem, st>>>(m[0], m[1], m[2], m[3], m[4],
                                                                      a);
  return cudaGetLastError();
}

template <int D, int DP>
cudaError_t launch_bwd_g(const Shape& s, const CUtensorMap* m, const BwdArgs& a, cudaStream_t st) {
  switch (s.G) {
    case 1: return launch_bwd_t<D, 1, DP>(s, m, a, st);
    case 2: return launch_bwd_t<D, 2, DP>(s, m, a, st);
    case 4: return launch_bwd_t<D, 4, DP>(s, m, a, st);
    default: return launch_bwd_t<D, 8, DP>(s, m, a, st);
  }
}

}  // namespace

cudaError_t launch_bwd(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                       const int32_t* row_ptr, const uint32_t* ent, uint8_t* rec,
                       const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const uint16_t* q_p, const uint16_t* dO, const float* lse,
                       const float* dsum, const float* mass, const float* sel_score,
                       const uint8_t* sel_arg, const float* plse, float* dq_part, float* dk,
                       float* dv, float* dk_p, unsigned* status, cudaStream_t st) {
  CUtensorMap m[5];
  cudaError_t e;
  if ((e = make_tmap_3d(&m[0], q, s.d, s.hq, s.T, 64, s.G, 1, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&m[1], dO, s.d, s.hq, s.T, 64, s.G, 1, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&m[2], k, s.d, s.hkv, s.T, 64, 1, 128, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&m[3], v, s.d, s.hkv, s.T, 64, 1, 128, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&m[4], q_p, s.dp, s.hkv, s.T, s.dp, 1, 1, 0)) != cudaSuccess) return e;
  BwdArgs a{cu_seqlens, cu_blocks, row_ptr,    ent,        rec,          lse,         dsum,
            mass,       sel_score, sel_arg,    plse,       s.ndoc,       s.T,         s.hq,
            s.hkv,      s.K,       s.nb_bound, s.softmax_scale, s.proxy_scale, s.kl_weight,
            dq_part,    dk,        dv,         dk_p,       status};
  if (s.d == 128)
    return s.dp == 64 ? launch_bwd_g<128, 64>(s, m, a, st) : launch_bwd_g<128, 32>(s, m, a, st);
  return s.dp == 64 ? launch_bwd_g<64, 64>(s, m, a, st) : launch_bwd_g<64, 32>(s, m, a, st);
}

}  // namespace msa
