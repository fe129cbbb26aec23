// Proxy scoring with on-chip 128-key block max-pool and streaming top-k.
//
// The proxy head scores every causal key; KV is then chosen in 128-token
// blocks by the maximum proxy score inside each block ("Dramatically Speeding
// Up Million-Token Training! ... 'Flash-MSA' ...", ai-minor.com, "What's
// Happening? News Overview"), each query keeping its top-k blocks with its own
// diagonal block always included.
//
// One CTA per (query block J of a document, KV group g).  For every key block
// n = 0..J the tensor cores compute the 128x128 score tile q_p . k_p^T into
// TMEM (K = dp), and the epilogue threads (one TMEM lane = one query row)
// reduce it to the block maximum and, when the block enters the row's top
// list, its lowest-index argmax.  Neither the score tile nor the pooled
// [T, blocks] matrix ever leaves the SM.
//
// Roles (512 threads): warps 0-11 are three epilogue warpgroups, warp 12
// issues TMA loads of k_p into a ring, warp 13 issues tcgen05.mma, warps 14-15
// idle.  Key blocks go in steps of two: one 256-row k_p box per step, one
// N = 256 MMA chain into one of two 256-column TMEM accumulators (steps
// alternate), so the fixed cost of a step (barrier hand-offs, commits) is paid
// once per two blocks.  Block n goes to epilogue warpgroup n mod 3: three
// warpgroups keep the max trees of the blocks fed to the tensor core (with two,
// the tensor pipe waited on the epilogue more than half of the time), and a
// step's accumulator is released once both of its blocks have been read.
// Register budgets per warpgroup: 3 x 128 x 152 (epilogue) + 128 x 56 = 65536.
//
// Block pattern: with a window (w, s) the blocks J - s*u, u = 1..w, are kept
// whatever their score; the pattern is configurable by window size and
// dilation ("Flash-MSA: Ein Training mit einer Million Tokens ohne hohe
// Rechenkosten", keelcrux.com, "Under the hood").  Their scores and argmaxes
// go to slots of their own in shared memory, they never enter the ranked list,
// and the ranked list fills the other k-1-|window| slots.
#include <cfloat>
#include <climits>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelEpiGroups = 3;
constexpr int kSelProducerWarp = 12, kSelMmaWarp = 13;
constexpr uint32_t kSelRegsEpi = 152, kSelRegsCtl = 56;
constexpr float kTieBand = 1e-3f;
// CTAs per cluster: query blocks gb0, gb0 - 1, ... of one group, which share
// their key blocks' k_p rows by multicast (2 or 4).  Four measured slower at
// 128k-1M: at most 36 clusters of four are resident, 144 of the 152 SMs.
constexpr int kSelCluster = 2;

// k_p ring stages (two key blocks each).  The TMA latency of a stage is about
// 3000 SM cycles at 128k, three steps' worth; six stages measured no faster.
template <bool WIN>
constexpr int sel_stages() { return 4; }

template <int DP>
struct SelCfg {
  static constexpr int kRowBytes = DP * 2;
  static constexpr int kTileBytes = 128 * kRowBytes;
  static constexpr uint32_t kLayout = DP == 64 ? kLayoutSW128 : kLayoutSW64;
  static constexpr uint32_t kSBO = 8 * kRowBytes;
};

// a ranks ahead of b: higher score, ties to the lower block id (id = block << 8 | arg)
__device__ __forceinline__ bool better(float sa, uint32_t ia, float sb, uint32_t ib) {
  return sa > sb || (sa == sb && (ia >> 8) < (ib >> 8));
}

// Insert (s, nid) into the descending list sc/id (CAP entries), dropping the last.
template <int CAP>
__device__ __forceinline__ void list_insert(float (&sc)[CAP], uint32_t (&id)[CAP], float s,
                                            uint32_t nid) {
  bool shift = false;
  float cs = s;
  uint32_t ci = nid;
#pragma unroll
  for (int i = 0; i < CAP; ++i) {
    const bool take = shift || better(s, nid, sc[i], id[i]);
    const float ts = sc[i];
    const uint32_t ti = id[i];
    sc[i] = take ? cs : ts;
    id[i] = take ? ci : ti;
    cs = take ? ts : cs;
    ci = take ? ti : ci;
    shift = take;
  }
}

// Insert (s, nid) into the descending list sc/id when every entry already in
// the list came from a lower block id: an equal score never displaces an
// entry, so "ranks ahead" is a strict score comparison.  The list is sorted,
// so the flags s > sc[i] switch from false to true once; entry i becomes
// sc[i-1] after that point, s at it, and stays itself before it.
template <int CAP>
__device__ __forceinline__ void list_insert_newer(float (&sc)[CAP], uint32_t (&id)[CAP], float s,
                                                  uint32_t nid) {
  bool prev = false;
  float ps = 0.f;
  uint32_t pi = 0u;
#pragma unroll
  for (int i = 0; i < CAP; ++i) {
    const bool cur = s > sc[i];
    const float os = sc[i];
    const uint32_t oi = id[i];
    sc[i] = prev ? ps : (cur ? s : os);
    id[i] = prev ? pi : (cur ? nid : oi);
    ps = os;
    pi = oi;
    prev = cur;
  }
}

// Maximum of 32 scores held as raw fp32 bits (16 three-input max instructions).
__device__ __forceinline__ float max32(const uint32_t (&r)[32]) {
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

struct SelArgs {
  const int32_t* cu;
  const int32_t* cu_blocks;
  int ndoc, T, hkv, K, nb_bound;
  int window, dilation;  // always-kept blocks J - dilation * u, u = 1..window
  float proxy_scale;
  int32_t* sel_idx;
  float* sel_score;
  uint8_t* sel_arg;
  float* plse;
  uint8_t* tie;
  unsigned* status;
  bool withhold_q;  // test hook: never load the query tile (the MMA warp's wait runs out)
};

template <int DP, int CAP, bool ARG, bool WIN>
__global__ void __launch_bounds__(kSelThreads, 1)
    k_select(const __grid_constant__ CUtensorMap tm_qp, const __grid_constant__ CUtensorMap tm_kp,
             const SelArgs a) {
  using C = SelCfg<DP>;
  constexpr int kSelStages = sel_stages<WIN>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  // ---- shared memory carve-up ----
  uint8_t* sQ = smem;                                   // q_p tile, 128 rows
  uint8_t* sK = sQ + C::kTileBytes;                     // k_p ring: pairs of 128-key blocks
  // lists of warpgroups 1 and 2 for the merge, [2][CAP][128]: in the k_p ring,
  // which is free by then
  float* m_sc = reinterpret_cast<float*>(sK);
  uint32_t* m_id = reinterpret_cast<uint32_t*>(m_sc + 2 * CAP * 128);
  static_assert(2 * CAP * 128 * 8 <= kSelStages * 2 * C::kTileBytes, "merge lists fit the ring");
  float* d_sc = reinterpret_cast<float*>(sK + kSelStages * 2 * C::kTileBytes);  // [128]
  uint32_t* d_id = reinterpret_cast<uint32_t*>(d_sc + 128);                 // [128]
  // [CAP][128] always-kept blocks (block pattern only)
  float* f_sc = reinterpret_cast<float*>(d_id + 128);
  uint32_t* f_id = reinterpret_cast<uint32_t*>(f_sc + (WIN ? CAP * 128 : 0));
  uint64_t* bars = reinterpret_cast<uint64_t*>(f_id + (WIN ? CAP * 128 : 0));
  // bars: 0 qfull | 1..S kvfull | S+1..2S kvempty | 2S+1..2S+2 accfull | 2S+3..2S+4 accempty
  // | 2S+5 MMAs done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2 * kSelStages + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  const uint32_t b_qfull = smem_u32(bars);
  auto b_kvfull = [&](int s) { return smem_u32(bars + 1 + s); };
  auto b_kvempty = [&](int s) { return smem_u32(bars + 1 + kSelStages + s); };
  auto b_accfull = [&](int i) { return smem_u32(bars + 1 + 2 * kSelStages + i); };
  auto b_accempty = [&](int i) { return smem_u32(bars + 3 + 2 * kSelStages + i); };
  const uint32_t b_mmadone = smem_u32(bars + 5 + 2 * kSelStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item.  A cluster of kSelCluster CTAs takes query blocks gb0,
  // gb0 - 1, ... of group g (heaviest first); CTA `rank` takes gb0 - rank.
  // When all of them lie in one document (shared), their first key blocks
  // are the same k_p rows: each of a step's two key blocks is loaded by one
  // CTA and multicast to all, so the cluster reads k_p from L2 once instead
  // of kSelCluster times.  With two CTAs, rank r loads block 2m + r of step
  // m; with four, ranks 0-1 load the blocks of even steps, ranks 2-3 those
  // of odd steps. ----
  const uint32_t rank = cluster_ctarank();
  const bool ok_batch = a.cu_blocks[a.ndoc + 1] != 0;  // else malformed cu_seqlens (flagged by k_meta)
  const int nbt = min(a.cu_blocks[a.ndoc], a.nb_bound);
  const int cl = (int)(blockIdx.x / kSelCluster);
  const int g = cl % a.hkv;
  const int gb0 = nbt - 1 - kSelCluster * (cl / a.hkv);
  const int gb = gb0 - (int)rank;
  const bool has = ok_batch && gb >= 0;  // warp- and CTA-uniform
  const bool shared_kp = ok_batch && gb0 >= kSelCluster - 1 &&
                      doc_of_block(a.cu_blocks, a.ndoc, gb0) ==
                          doc_of_block(a.cu_blocks, a.ndoc, gb0 - (kSelCluster - 1));
  const int d = has ? doc_of_block(a.cu_blocks, a.ndoc, gb) : 0;
  const int J = has ? gb - a.cu_blocks[d] : 0;
  const int dstart = has ? a.cu[d] : 0;
  const int L = has ? a.cu[d + 1] - dstart : 0;
  const int qstart = dstart + J * kBlock;
  const int nrows = min(kBlock, L - J * kBlock);
  const int nblk = has ? J + 1 : 0;
  const int nstep = (nblk + 1) / 2;  // steps of two key blocks (the last may hold one)
  // Steps every CTA of the cluster takes (the last rank's count, with J0 =
  // J + rank the first rank's block; lower ranks load their one or two extra
  // steps alone); 0 when not shared.
  const int common = shared_kp ? (J + (int)rank - (kSelCluster - 1) + 2) / 2 : 0;
  constexpr uint16_t kMcMask = (uint16_t)((1u << kSelCluster) - 1);

  if (threadIdx.x == 0) {
    mbar_init(b_qfull, 1);
    for (int s = 0; s < kSelStages; ++s) {
      mbar_init(b_kvfull(s), 1);
      mbar_init(b_kvempty(s), shared_kp ? kSelCluster : 1);  // a shared stage: every CTA's MMA warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_accfull(i), 1);
      mbar_init(b_accempty(i), 8);  // four warps for each of the step's two blocks
    }
    mbar_init(b_mmadone, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (has && warp == kSelMmaWarp) {
    tmem_alloc(smem_u32(tslot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the peer's barriers are initialised before any multicast copy or commit
  // reaches them
  cluster_sync();
  const uint32_t tbase = has ? *reinterpret_cast<volatile uint32_t*>(tslot) : 0u;

  if (!has) {
    // no query block for this CTA: nothing but the cluster barrier below
  } else if (warp >= 4 * kSelEpiGroups) {
    setmaxnreg_dec<kSelRegsCtl>();
    if (warp == kSelProducerWarp) {
      // ------------------------------ TMA producer ------------------------------
      if (lane == 0) {
        tma_prefetch_desc(&tm_qp);
        tma_prefetch_desc(&tm_kp);
        if (!a.withhold_q) {
          mbar_arrive_expect_tx(b_qfull, C::kTileBytes);
          tma_load_3d(smem_u32(sQ), &tm_qp, b_qfull, 0, g, qstart);
        }
        // step m: key blocks 2m and 2m+1 as one 256-row box (rows past the
        // diagonal block, or past T, are loaded or zero-filled and never read)
        int issued = 0;
        for (int m = 0; m < nstep; ++m) {
          const int s = m % kSelStages;
          if (m >= kSelStages &&
              !wait_bar(b_kvempty(s), ((m / kSelStages) & 1) ^ 1, abort_flag, a.status,
                        wait_site(kKerSelect, 7 + s, m)))
            break;
          mbar_arrive_expect_tx(b_kvfull(s), 2 * C::kTileBytes);
          const uint32_t dst = smem_u32(sK + s * 2 * C::kTileBytes);
          if (m < common) {  // this CTA's key block of the step, if any, for every CTA
            const int u = (int)(rank & 1);
            if (kSelCluster == 2 || (int)(rank >> 1) == (m & 1))
              tma_load_3d_mc(dst + u * C::kTileBytes, &tm_kp, b_kvfull(s), 0, g,
                             dstart + (2 * m + u) * kBlock, kMcMask);
          } else {
            tma_load_3d(dst, &tm_kp, b_kvfull(s), 0, g, dstart + 2 * m * kBlock);
            tma_load_3d(dst + C::kTileBytes, &tm_kp, b_kvfull(s), 0, g,
                        dstart + (2 * m + 1) * kBlock);
          }
          issued = m + 1;
        }
        // Let this CTA's own copies land before it exits (they have, unless a
        // wait gave up): the last use of every ring stage, and the query tile.
        for (int m = issued > kSelStages ? issued - kSelStages : 0; m < issued; ++m)
          drain_bar(b_kvfull(m % kSelStages), (m / kSelStages) & 1);
        if (!a.withhold_q) drain_bar(b_qfull, 0);
      }
    } else if (warp == kSelMmaWarp) {
      // ------------------------------ MMA issuer ---------------------------------
      if (lane == 0) {
        constexpr uint32_t idesc = make_idesc_bf16(128, 256, false, false);
        if (wait_bar(b_qfull, 0, abort_flag, a.status, wait_site(kKerSelect, 0, 0))) {
          const uint32_t q0 = smem_u32(sQ);
          for (int m = 0; m < nstep; ++m) {
            const int s = m % kSelStages, acc = m & 1;
            if (!wait_bar(b_kvfull(s), (m / kSelStages) & 1, abort_flag, a.status,
                          wait_site(kKerSelect, 1 + s, m)))
              break;
            if (m >= 2 && !wait_bar(b_accempty(acc), ((m >> 1) & 1) ^ 1, abort_flag, a.status,
                                    wait_site(kKerSelect, 17 + acc, m)))
              break;
            tc_fence_after();
            const uint32_t k0 = smem_u32(sK + s * 2 * C::kTileBytes);
            // scores of 128 queries x 256 keys (two blocks) into a 256-column accumulator
#pragma unroll
            for (int kk = 0; kk < DP / 16; ++kk) {
              const uint64_t ad = make_sdesc(q0 + kk * 32, 16, C::kSBO, C::kLayout);
              const uint64_t bd = make_sdesc(k0 + kk * 32, 16, C::kSBO, C::kLayout);
              umma_bf16(tbase + acc * 256, ad, bd, idesc, kk > 0);
            }
            if (m < common) umma_commit_mc(b_kvempty(s), kMcMask);  // every CTA's copy of the stage
            else umma_commit(b_kvempty(s));
            umma_commit(b_accfull(acc));
          }
        }
        // every MMA issued by this CTA completes before TMEM is released
        umma_commit(b_mmadone);
        drain_bar(b_mmadone, 0);
      }
    }
  } else {
    setmaxnreg_inc<kSelRegsEpi>();
    // ------------------------------ epilogue -----------------------------------
    const int e = warp >> 2;            // warpgroup 0, 1 or 2
    const int row = (warp & 3) * 32 + lane;  // TMEM lane = query row in the block
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float sc[CAP];
    uint32_t id[CAP];
#pragma unroll
    for (int i = 0; i < CAP; ++i) {
      sc[i] = -FLT_MAX;
      id[i] = 0xFFFFFFFFu;
    }
    float dsv = -FLT_MAX;
    uint32_t dav = 0;
    bool handled_diag = false;
    const float ps = a.proxy_scale;
    // Always-kept blocks J - dilation * u, u = min(window, J / dilation) .. 1: the
    // lowest one, then a cursor this warpgroup advances as its blocks (in
    // increasing order) pass it, so the block loop needs no division.
    int next_kept = INT_MAX;
    if (WIN && J >= a.dilation) next_kept = J - a.dilation * min(a.window, J / a.dilation);
    // Warpgroup e takes the blocks n = e, e + 3, ... in increasing order; block
    // n sits in half n & 1 of accumulator (n >> 1) & 1.
#pragma unroll 1
    for (int n = e; n < nblk; n += kSelEpiGroups) {
      const int m = n >> 1, acc = m & 1, u = n & 1;
      if (!wait_bar_warp(b_accfull(acc), (m >> 1) & 1, abort_flag, a.status,
                         wait_site(kKerSelect, 13 + acc, m)))
        break;
      tc_fence_after();
      const uint32_t tb = tbase + lane_off + acc * 256 + u * 128;
      const bool diag = (n == J);
      // block of the always-kept window (warp-uniform)
      bool forced = false;
      if (WIN && !diag && n >= next_kept) {
        while (next_kept < n) next_kept += a.dilation;
        forced = n == next_kept;
      }
      // argmax bookkeeping for every block (ARG), else for the diagonal block only
      const bool track = ARG || diag;  // warp-uniform
      // The 32 scores of the chunk holding the row maximum stay in registers (first chunk
      // on ties), so the argmax needs no second TMEM read.
      uint32_t bv[32];
      float best = 0.f;
      int bc = 0;
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {  // 64 columns per TMEM round trip
        uint32_t va[32], vb[32];
        tmem_ld32x2(tb + c2 * 64, tb + c2 * 64 + 32, va, vb);
        if (c2 == 1) {  // the block's scores are all in registers: release its accumulator half
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_accempty(acc));
        }
        if (diag) {
          const uint32_t neg = __float_as_uint(-FLT_MAX);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (c2 * 64 + i > row) va[i] = neg;
            if (c2 * 64 + 32 + i > row) vb[i] = neg;
          }
        }
        const float ma = max32(va), mb = max32(vb);
        if (c2 == 0) {
          const bool tb1 = mb > ma;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (track) bv[i] = tb1 ? vb[i] : va[i];
          best = tb1 ? mb : ma;
          bc = tb1 ? 1 : 0;
        } else {
          const bool ta = ma > best;
          const float m2 = ta ? ma : best;
          const bool tb1 = mb > m2;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (track) bv[i] = tb1 ? vb[i] : (ta ? va[i] : bv[i]);
          best = tb1 ? mb : m2;
          bc = tb1 ? 3 : (ta ? 2 : bc);
        }
      }
      // blocks reach this warpgroup in increasing order, so ties keep the older entry
      const bool need = diag || forced || best * ps > sc[CAP - 1];
      int arg = 0;
      if (need && track) {
        int aa = 31;
#pragma unroll
        for (int i = 30; i >= 0; --i) aa = (__uint_as_float(bv[i]) == best) ? i : aa;
        arg = bc * 32 + aa;
      }
      if (diag) {
        dsv = best * ps;
        dav = ((uint32_t)n << 8) | (uint32_t)arg;
        handled_diag = true;
      } else if (forced) {  // kept whatever its score: a slot of its own, not the ranking
        const int u = (J - n) / a.dilation - 1;
        f_sc[u * 128 + row] = best * ps;
        f_id[u * 128 + row] = ((uint32_t)n << 8) | (uint32_t)arg;
      } else if (need) {
        list_insert_newer<CAP>(sc, id, best * ps, ((uint32_t)n << 8) | (uint32_t)arg);
      }
    }
    // ---- merge the lists of warpgroups 1 and 2 into warpgroup 0's ----
    if (handled_diag) {
      d_sc[row] = dsv;
      d_id[row] = dav;
    }
    // every warpgroup has read its last scores: every MMA and so every k_p
    // load has completed, and the lists can go into the ring
    named_bar_sync(1, 128 * kSelEpiGroups);
    if (e >= 1) {
#pragma unroll
      for (int i = 0; i < CAP; ++i) {
        m_sc[((e - 1) * CAP + i) * 128 + row] = sc[i];
        m_id[((e - 1) * CAP + i) * 128 + row] = id[i];
      }
    }
    named_bar_sync(1, 128 * kSelEpiGroups);
    if (e == 0) {
#pragma unroll 1
      for (int w = 0; w < kSelEpiGroups - 1; ++w) {
#pragma unroll
        for (int i = 0; i < CAP; ++i) {
          const uint32_t oid = m_id[(w * CAP + i) * 128 + row];
          if (oid != 0xFFFFFFFFu) list_insert<CAP>(sc, id, m_sc[(w * CAP + i) * 128 + row], oid);
        }
      }
      dsv = d_sc[row];
      dav = d_id[row];
      const int K = a.K;
      const int nsel = min(J, K - 1);  // off-diagonal blocks kept
      const int nf = WIN ? min(a.window, J / a.dilation) : 0;  // always kept
      const int ntop = nsel - nf;      // chosen by score from the other earlier blocks
      uint8_t tie = 0;
      if (J > K - 1 && ntop >= 1) {  // a choice was made: last taken vs first left
        float s_last = 0.f, s_next = 0.f;
#pragma unroll
        for (int i = 0; i < CAP; ++i) {
          if (i == ntop - 1) s_last = sc[i];
          if (i == ntop) s_next = sc[i];
        }
        tie = (s_last - s_next) < kTieBand ? 1 : 0;
      }
      // the always-kept blocks take list entries ntop .. nsel-1
#pragma unroll
      for (int i = 0; i < CAP; ++i) {
        if (WIN && i >= ntop && i < nsel) {
          sc[i] = f_sc[(i - ntop) * 128 + row];
          id[i] = f_id[(i - ntop) * 128 + row];
        }
      }
      // plse over the selection (nsel best + diagonal)
      float mx = dsv;
#pragma unroll
      for (int i = 0; i < CAP; ++i)
        if (i < nsel) mx = fmaxf(mx, sc[i]);
      float se = __expf(dsv - mx);
#pragma unroll
      for (int i = 0; i < CAP; ++i)
        if (i < nsel) se += __expf(sc[i] - mx);
      const float plse_v = mx + __logf(se);
      // ascending block order of the nsel kept entries (odd-even transposition)
      uint32_t key[CAP];
#pragma unroll
      for (int i = 0; i < CAP; ++i) key[i] = i < nsel ? (id[i] >> 8) : 0xFFFFFFFFu;
#pragma unroll
      for (int p = 0; p < CAP; ++p) {
#pragma unroll
        for (int i = (p & 1); i + 1 < CAP; i += 2) {
          const bool sw = key[i] > key[i + 1];
          const uint32_t k0 = key[i], k1 = key[i + 1], i0 = id[i], i1 = id[i + 1];
          const float s0 = sc[i], s1 = sc[i + 1];
          key[i] = sw ? k1 : k0;
          key[i + 1] = sw ? k0 : k1;
          id[i] = sw ? i1 : i0;
          id[i + 1] = sw ? i0 : i1;
          sc[i] = sw ? s1 : s0;
          sc[i + 1] = sw ? s0 : s1;
        }
      }
      const int t = qstart + row;
      // a CTA whose waits gave up leaves the outputs untouched
      if (row < nrows && t < a.T && !*abort_flag) {
        const size_t base = ((size_t)t * a.hkv + g) * K;
#pragma unroll
        for (int s = 0; s < kMaxTopK; ++s) {
          if (s >= K) break;
          int32_t b = -1;
          float scv = 0.f;
          uint8_t av = 0;
#pragma unroll
          for (int i = 0; i < CAP; ++i)
            if (i == s && i < nsel) {
              b = (int32_t)(id[i] >> 8);
              scv = sc[i];
              av = (uint8_t)(id[i] & 0xFF);
            }
          if (s == nsel) {
            b = J;
            scv = dsv;
            av = (uint8_t)(dav & 0xFF);
          }
          a.sel_idx[base + s] = b;
          a.sel_score[base + s] = scv;
          a.sel_arg[base + s] = av;
        }
        a.plse[(size_t)t * a.hkv + g] = plse_v;
        a.tie[(size_t)t * a.hkv + g] = tie;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (has && warp == kSelMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  // neither CTA leaves while the other may still copy into its shared memory
  // or arrive on its barriers
  cluster_sync();
}

template <int DP, int CAP, bool ARG, bool WIN>
cudaError_t launch_sel_t(const Shape& s, const CUtensorMap& mq, const CUtensorMap& mk,
                         const SelArgs& a, cudaStream_t st) {
  using C = SelCfg<DP>;
  constexpr int kSelStages = sel_stages<WIN>();
  const size_t smem = 1024 + (1 + 2 * kSelStages) * C::kTileBytes + (WIN ? CAP * 128 * 8 : 0) +
                      128 * 8 + (2 * kSelStages + 6) * 8 + 16;
  static_assert(1024 + (1 + 2 * kSelStages) * SelCfg<64>::kTileBytes + (WIN ? 16 * 128 * 8 : 0) +
                        128 * 8 + (2 * kSelStages + 6) * 8 + 16 <= 232448,
                "shared memory budget");
  // The warpgroups' register budgets are drawn from the registers the block
  // is launched with; a larger sum would leave setmaxnreg.inc waiting.
  constexpr int kBudget = kSelEpiGroups * 128 * kSelRegsEpi + 128 * kSelRegsCtl;
  static_assert(kBudget <= 65536, "register budgets exceed the register file");
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, k_select<DP, CAP, ARG, WIN>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kSelThreads < kBudget) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(k_select<DP, CAP, ARG, WIN>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // clusters of kSelCluster CTAs: query blocks gb0, gb0 - 1, ... of one group
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim =
      dim3((unsigned)(kSelCluster * s.hkv * ((s.nb_bound + kSelCluster - 1) / kSelCluster)));
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSelCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_select<DP, CAP, ARG, WIN>, mq, mk, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The block pattern is a template switch: without it the block loop and the
// merge compile exactly as the plain rule needs.
template <int DP, int CAP>
cudaError_t launch_sel_a(const Shape& s, const CUtensorMap& mq, const CUtensorMap& mk,
                         const SelArgs& a, bool with_arg, cudaStream_t st) {
  if (s.window > 0)
    return with_arg ? launch_sel_t<DP, CAP, true, true>(s, mq, mk, a, st)
                    : launch_sel_t<DP, CAP, false, true>(s, mq, mk, a, st);
  return with_arg ? launch_sel_t<DP, CAP, true, false>(s, mq, mk, a, st)
                  : launch_sel_t<DP, CAP, false, false>(s, mq, mk, a, st);
}

}  // namespace

cudaError_t launch_select(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                          const uint16_t* q_p, const uint16_t* k_p, int32_t* sel_idx,
                          float* sel_score, uint8_t* sel_arg, float* plse, uint8_t* tie,
                          bool with_arg, unsigned* status, cudaStream_t st) {
  CUtensorMap mq, mk;
  const int sw = s.dp == 64 ? 128 : 64;
  cudaError_t e;
  if ((e = make_tmap_3d(&mq, q_p, s.dp, s.hkv, s.T, s.dp, 1, 128, sw)) != cudaSuccess) return e;
  // one 128-row key block per box (a step loads two, or each loading CTA of a cluster one)
  if ((e = make_tmap_3d(&mk, k_p, s.dp, s.hkv, s.T, s.dp, 1, 128, sw)) != cudaSuccess) return e;
  SelArgs a{cu_seqlens, cu_blocks, s.ndoc,   s.T,         s.hkv, s.K,
            s.nb_bound, s.window,  s.dilation, s.proxy_scale, sel_idx, sel_score,
            sel_arg,    plse,      tie,    status, s.test_stall_select};
  const int cap = s.K <= 4 ? 4 : (s.K <= 8 ? 8 : 16);
  if (s.dp == 64) {
    if (cap == 4) return launch_sel_a<64, 4>(s, mq, mk, a, with_arg, st);
    if (cap == 8) return launch_sel_a<64, 8>(s, mq, mk, a, with_arg, st);
    return launch_sel_a<64, 16>(s, mq, mk, a, with_arg, st);
  }
  if (cap == 4) return launch_sel_a<32, 4>(s, mq, mk, a, with_arg, st);
  if (cap == 8) return launch_sel_a<32, 8>(s, mq, mk, a, with_arg, st);
  return launch_sel_a<32, 16>(s, mq, mk, a, with_arg, st);
}

}  // namespace msa
