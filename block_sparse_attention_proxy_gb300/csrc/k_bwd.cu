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
// Fused proxy part: every gathered (token, slot) carries
//   g_b = kl_weight * proxy_scale * (exp(S_b - plse) - m_b),
// and dk_p[a_b] += g_b q_p[t] is accumulated in shared memory for the block's
// 128 keys in a fixed order by one warp, then written once.
//
// Roles (224 threads): warps 0-3 epilogue, warp 4 TMA producer + row metadata,
// warp 5 MMA issuer, warp 6 proxy-gradient accumulator.
#include <cfloat>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kBwdThreads = 224;
constexpr int kRT = 64;  // rows per tile
constexpr float kLog2eB = 1.4426950408889634f;

struct BwdArgs {
  const int32_t* cu;
  const int32_t* cu_blocks;
  const int32_t* row_ptr;
  const uint32_t* ent;
  const uint16_t* q_p;
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

struct RowMeta {
  float lse[kRT];
  float dsum[kRT];
  int32_t qpos[kRT];
  int32_t t[kRT];
  int32_t hs[kRT];  // head | slot << 8
  int32_t tok_t[kRT];
  int32_t tok_a[kRT];
  float tok_g[kRT];
};

template <int D, int G, int DP>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_bwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
          const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
          const BwdArgs a) {
  constexpr int TPT = kRT / G;
  constexpr int NCH = D / 64;
  constexpr int kKV = 128 * D * 2;
  constexpr int kQT = kRT * D * 2;
  constexpr int kQChunk = kRT * 128;  // bytes of one 64-column chunk of a 64-row tile
  constexpr uint32_t T_S = 0, T_DP = 64, T_DV = 128, T_DK = 128 + D, T_DQ = 128 + 2 * D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + kKV;
  uint8_t* sQ = sV + kKV;         // [2]
  uint8_t* sdO = sQ + 2 * kQT;    // [2]
  uint8_t* sPs = sdO + 2 * kQT;   // [128 keys][64 rows] bf16, 128B swizzle
  uint8_t* sdS = sPs + 16384;     // [128 keys][64 rows] hi part of dS
  uint8_t* sdSl = sdS + 16384;    // [128 keys][64 rows] lo part of dS
  // sPs..sdS (32 KB) double as the fp32 dQ stage [64 rows][D] once a tile's MMAs are done
  float* sdkp = reinterpret_cast<float*>(sdSl + 16384);     // [128][DP]
  RowMeta* meta = reinterpret_cast<RowMeta*>(sdkp + 128 * DP);  // [2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(meta + 2);
  // 0 kv_full | 1,2 q_full | 3,4 tile_done | 5 sp_full | 6 ds_full | 7 dq_full
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 8);
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
  const int lbeg = a.row_ptr[g * a.nb_bound + gb];
  const int lcnt = a.row_ptr[g * a.nb_bound + gb + 1] - lbeg;
  const int ndiag = (nkeys + TPT - 1) / TPT;
  const int ntiles = ndiag + (lcnt + TPT - 1) / TPT;
  const int slot_diag = min(j, a.K - 1);

  if (threadIdx.x == 0) {
    mbar_init(bar(0), 1);
    mbar_init(bar(1), 1);
    mbar_init(bar(2), 1);
    mbar_init(bar(3), 5);
    mbar_init(bar(4), 5);
    mbar_init(bar(5), 1);
    mbar_init(bar(6), 4);
    mbar_init(bar(7), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tslot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(tslot);

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

  if (warp == 4) {
    // ------------------------- TMA producer + row metadata ------------------------
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(0), 2 * kKV);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        tma_load_3d(smem_u32(sK + c * 16384), &tm_k, bar(0), 64 * c, g, kstart);
        tma_load_3d(smem_u32(sV + c * 16384), &tm_v, bar(0), 64 * c, g, kstart);
      }
    }
    const float gscale = a.kl_weight * a.proxy_scale;
    for (int n = 0; n < ntiles; ++n) {
      const int buf = n & 1;
      if (n >= 2 && !wait_bar_warp(bar(3 + buf), ((n >> 1) & 1) ^ 1, abort_flag, a.status,
                                   wait_site(kKerBwd, 3 + buf, n)))
        break;
      RowMeta& m = meta[buf];
      const bool diag = n < ndiag;
      // per token (lane < TPT): proxy-gradient coefficient
      for (int i = lane; i < TPT; i += 32) {
        int t, slot;
        const bool valid = tile_token(n, i, t, slot);
        float gs = 0.f;
        int arg = 0;
        if (valid) {
          const size_t e = ((size_t)t * a.hkv + g) * a.K + slot;
          const float p = __expf(__ldg(a.sel_score + e) - __ldg(a.plse + (size_t)t * a.hkv + g));
          gs = gscale * (p - __ldg(a.mass + e));
          arg = __ldg(a.sel_arg + e) & (kBlock - 1);  // in-block offset; keeps smem indexing in range
        }
        m.tok_t[i] = valid ? t : -1;
        m.tok_a[i] = arg;
        m.tok_g[i] = gs;
      }
      // per row (two per lane)
      for (int r = lane; r < kRT; r += 32) {
        const int i = r / G, hl = r % G;
        int t, slot;
        const bool valid = tile_token(n, i, t, slot);
        const size_t row = (size_t)t * a.hq + g * G + hl;
        m.lse[r] = valid ? __ldg(a.lse + row) : __int_as_float(0x7f800000);  // +inf -> P = 0
        m.dsum[r] = valid ? __ldg(a.dsum + row) : 0.f;
        m.qpos[r] = diag ? n * TPT + i : (1 << 30);
        m.t[r] = valid ? t : -1;
        m.hs[r] = (g * G + hl) | (slot << 8);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(bar(1 + buf), 2 * kQT);
      __syncwarp();
      const uint32_t qb = smem_u32(sQ + buf * kQT), ob = smem_u32(sdO + buf * kQT);
      for (int i = lane; i < TPT; i += 32) {
        int t, slot;
        if (!tile_token(n, i, t, slot)) t = a.T;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          tma_load_3d(qb + c * kQChunk + i * G * 128, &tm_q, bar(1 + buf), 64 * c, g * G, t);
          tma_load_3d(ob + c * kQChunk + i * G * 128, &tm_do, bar(1 + buf), 64 * c, g * G, t);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------ MMA issuer ---------------------------------
    if (lane == 0) {
      constexpr uint32_t idST = make_idesc_bf16(128, kRT, false, false);
      constexpr uint32_t idDV = make_idesc_bf16(128, D, false, true);
      constexpr uint32_t idDQ = make_idesc_bf16(128, kRT, true, true);
      bool ok = wait_bar(bar(0), 0, abort_flag, a.status, wait_site(kKerBwd, 0, 0));
      const uint32_t k0 = smem_u32(sK), v0 = smem_u32(sV);
      const uint32_t ps0 = smem_u32(sPs), ds0 = smem_u32(sdS), dl0 = smem_u32(sdSl);
      for (int n = 0; ok && n < ntiles; ++n) {
        const int buf = n & 1, ph = (n >> 1) & 1;
        if (!wait_bar(bar(1 + buf), ph, abort_flag, a.status, wait_site(kKerBwd, 1 + buf, n)))
          break;
        if (n >= 1 && !wait_bar(bar(3 + ((n - 1) & 1)), ((n - 1) >> 1) & 1, abort_flag, a.status,
                                wait_site(kKerBwd, 3 + ((n - 1) & 1), n)))
          break;
        tc_fence_after();
        const uint32_t q0 = smem_u32(sQ + buf * kQT), o0 = smem_u32(sdO + buf * kQT);
        // S^T = K Q^T and dP^T = V dO^T   (M = 128 keys, N = 64 rows, K = D)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t kv_off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t q_off = (kk >> 2) * kQChunk + (kk & 3) * 32;
          umma_bf16(tbase + T_S, make_sdesc(k0 + kv_off, 16, 1024, kLayoutSW128),
                    make_sdesc(q0 + q_off, 16, 1024, kLayoutSW128), idST, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t kv_off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t q_off = (kk >> 2) * kQChunk + (kk & 3) * 32;
          umma_bf16(tbase + T_DP, make_sdesc(v0 + kv_off, 16, 1024, kLayoutSW128),
                    make_sdesc(o0 + q_off, 16, 1024, kLayoutSW128), idST, kk > 0);
        }
        umma_commit(bar(5));
        if (!wait_bar(bar(6), n & 1, abort_flag, a.status, wait_site(kKerBwd, 6, n))) break;
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
        umma_commit(bar(7));
      }
    }
  } else if (warp == 6) {
    // ------------------------ fused proxy gradient (dk_p) ------------------------
    constexpr int PER = DP / 32;
    for (int i = lane; i < 128 * DP; i += 32) sdkp[i] = 0.f;
    __syncwarp();
    for (int n = 0; n < ntiles; ++n) {
      const int buf = n & 1, ph = (n >> 1) & 1;
      if (!wait_bar_warp(bar(1 + buf), ph, abort_flag, a.status, wait_site(kKerBwd, 1 + buf, n)))
        break;
      const RowMeta& m = meta[buf];
      float x[TPT][PER];
#pragma unroll
      for (int i = 0; i < TPT; ++i) {
        const int t = m.tok_t[i];
#pragma unroll
        for (int u = 0; u < PER; ++u) x[i][u] = 0.f;
        if (t >= 0) {
          const uint16_t* src = a.q_p + ((size_t)t * a.hkv + g) * DP + lane * PER;
          if (PER == 2) {
            const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(src));
            x[i][0] = bf16_lo(w);
            x[i][PER - 1] = bf16_hi(w);
          } else {
            x[i][0] = __uint_as_float((uint32_t)__ldg(src) << 16);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < TPT; ++i) {
        if (m.tok_t[i] >= 0) {
          const float gs = m.tok_g[i];
          float* dst = sdkp + m.tok_a[i] * DP + lane * PER;
#pragma unroll
          for (int u = 0; u < PER; ++u) dst[u] = fmaf(gs, x[i][u], dst[u]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(3 + buf));
    }
    __syncwarp();
    for (int key = 0; key < nkeys; ++key) {
      float* dst = a.dk_p + ((size_t)(kstart + key) * a.hkv + g) * DP;
      for (int u = lane; u < DP; u += 32) dst[u] = sdkp[key * DP + u];
    }
  } else {
    // ------------------------------ epilogue ------------------------------------
    // Abort-safe: a failed wait marks the warp dead; it still walks every tile
    // and every named barrier so the other warps never wait on it forever.
    const int kk = warp * 32 + lane;  // key (S^T/dP^T/dV/dK lanes) or d index (dQ^T lanes)
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float sl2 = a.scale * kLog2eB;
    bool dead = false;
    for (int n = 0; n < ntiles; ++n) {
      const int buf = n & 1, ph = (n >> 1) & 1;
      const RowMeta& m = meta[buf];
      dead = dead || !wait_bar_warp(bar(1 + buf), ph, abort_flag, a.status,
                                    wait_site(kKerBwd, 1 + buf, n));
      dead = dead || !wait_bar_warp(bar(5), n & 1, abort_flag, a.status, wait_site(kKerBwd, 5, n));
      tc_fence_after();
      if (!dead) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // rows 32h .. 32h+31
          float s[32], dp[32];
          tmem_ld32f(tbase + lane_off + T_S + h * 32, s);
          tmem_ld32f(tbase + lane_off + T_DP + h * 32, dp);
          uint32_t pp[16], dh[16], dl[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float pv[2], hv[2], lv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int r = h * 32 + 2 * i + u;
              const float p = kk <= m.qpos[r]
                                  ? exp2f(fmaf(s[2 * i + u], sl2, -m.lse[r] * kLog2eB))
                                  : 0.f;
              const float ds = p * (dp[2 * i + u] - m.dsum[r]) * a.scale;
              pv[u] = p;
              hv[u] = __bfloat162float(__float2bfloat16_rn(ds));
              lv[u] = ds - hv[u];
            }
            pp[i] = pack_bf16(pv[0], pv[1]);
            dh[i] = pack_bf16(hv[0], hv[1]);
            dl[i] = pack_bf16(lv[0], lv[1]);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t off = sw128_offset((uint32_t)kk, (uint32_t)(h * 4 + q));
            *reinterpret_cast<uint4*>(sPs + off) =
                make_uint4(pp[4 * q], pp[4 * q + 1], pp[4 * q + 2], pp[4 * q + 3]);
            *reinterpret_cast<uint4*>(sdS + off) =
                make_uint4(dh[4 * q], dh[4 * q + 1], dh[4 * q + 2], dh[4 * q + 3]);
            *reinterpret_cast<uint4*>(sdSl + off) =
                make_uint4(dl[4 * q], dl[4 * q + 1], dl[4 * q + 2], dl[4 * q + 3]);
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(6));
      dead = dead || !wait_bar_warp(bar(7), n & 1, abort_flag, a.status, wait_site(kKerBwd, 7, n));
      tc_fence_after();
      // dQ^T: lane kk = head-dim index, 64 row columns -> fp32 stage [row][D] over sPs/sdS
      float* stage = reinterpret_cast<float*>(sPs);
      if (!dead) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float v[32];
          tmem_ld32f(tbase + lane_off + T_DQ + h * 32, v);
          if (kk < D) {
#pragma unroll
            for (int i = 0; i < 32; ++i) stage[(h * 32 + i) * D + kk] = v[i];
          }
        }
      }
      named_bar_sync(1, 128);
      constexpr int TPR = D / 4;            // threads per row (16 bytes each)
      constexpr int RPI = 128 / TPR;        // rows per iteration
      if (!dead) {
#pragma unroll 4
        for (int it = 0; it < kRT / RPI; ++it) {
          const int r = it * RPI + kk / TPR, c = kk % TPR;
          const int t = m.t[r];
          if (t >= 0) {
            const int hs = m.hs[r];
            float* dst = a.dq_part +
                         (((size_t)t * a.hq + (hs & 0xFF)) * a.K + (hs >> 8)) * (size_t)D + c * 4;
            *reinterpret_cast<float4*>(dst) =
                *reinterpret_cast<const float4*>(stage + r * D + c * 4);
          }
        }
      }
      named_bar_sync(1, 128);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(3 + buf));
    }
    // dK, dV rows of this block (lane = key), written once.  The TMEM loads are
    // warp-collective (.sync.aligned), so every lane of the warp executes them;
    // only the stores depend on the lane's key being inside the document.
    tc_fence_after();
    if (!dead) {
      const bool keep = kk < nkeys;
      float* dvr = a.dv + ((size_t)(kstart + (keep ? kk : 0)) * a.hkv + g) * D;
      float* dkr = a.dk + ((size_t)(kstart + (keep ? kk : 0)) * a.hkv + g) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32f(tbase + lane_off + T_DV + c * 32, v);
        if (keep) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(dvr + c * 32)[q] =
                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        tmem_ld32f(tbase + lane_off + T_DK + c * 32, v);
        if (keep) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(dkr + c * 32)[q] =
                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, int G, int DP>
cudaError_t launch_bwd_t(const Shape& s, const CUtensorMap* m, const BwdArgs& a, cudaStream_t st) {
  const size_t smem = 1024 + 2 * (128 * D * 2) + 4 * (kRT * D * 2) + 3 * 16384 +
                      128 * DP * 4 + 2 * sizeof(RowMeta) + 8 * 8 + 16;
  cudaError_t e = cudaFuncSetAttribute(k_bwd<D, G, DP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_bwd<D, G, DP><<<s.nb_bound * s.hkv, kBwdThreads, smem, st>>>(m[0], m[1], m[2], m[3], a);
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
                       const int32_t* row_ptr, const uint32_t* ent, const uint16_t* q,
                       const uint16_t* k, const uint16_t* v, const uint16_t* q_p,
                       const uint16_t* dO, const float* lse, const float* dsum, const float* mass,
                       const float* sel_score, const uint8_t* sel_arg, const float* plse,
                       float* dq_part, float* dk, float* dv, float* dk_p, unsigned* status,
                       cudaStream_t st) {
  CUtensorMap m[4];
  cudaError_t e;
  if ((e = make_tmap_3d(&m[0], q, s.d, s.hq, s.T, 64, s.G, 1, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&m[1], dO, s.d, s.hq, s.T, 64, s.G, 1, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&m[2], k, s.d, s.hkv, s.T, 64, 1, 128, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&m[3], v, s.d, s.hkv, s.T, 64, 1, 128, 128)) != cudaSuccess) return e;
  BwdArgs a{cu_seqlens, cu_blocks, row_ptr, ent,  q_p,  lse,   dsum,  mass,
            sel_score,  sel_arg,   plse,    s.ndoc, s.T, s.hq, s.hkv, s.K,
            s.nb_bound, s.softmax_scale, s.proxy_scale, s.kl_weight, dq_part, dk, dv, dk_p,
            status};
  if (s.d == 128)
    return s.dp == 64 ? launch_bwd_g<128, 64>(s, m, a, st) : launch_bwd_g<128, 32>(s, m, a, st);
  return s.dp == 64 ? launch_bwd_g<64, 64>(s, m, a, st) : launch_bwd_g<64, 32>(s, m, a, st);
}

}  // namespace msa
