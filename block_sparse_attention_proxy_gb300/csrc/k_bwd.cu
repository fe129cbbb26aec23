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
// Roles (512 threads): warps 0-7 softmax epilogue (two warpgroups, each half
// of a tile's rows), warps 8-11 dQ drain, warp 12 producer (Q/dO gathers by
// cp.async, records and q_p rows by bulk/TMA copies), warp 13 MMA issuer,
// warps 14-15 idle.  Two tiles are in flight: TMEM holds two slots of
// {S^T, dP^T}; after the epilogue has read a slot it writes P^T (bf16) back
// into the slot's dP^T columns, where the dV product reads it as its A
// operand, and the slot's S^T columns receive that tile's dQ^T.  dS^T has one shared-memory buffer: a tile's first dS^T
// store waits for the previous tile's products.  The MMA warp issues
// S^T/dP^T of tile n+1 ahead of the dV/dK/dQ products of tile n, so the
// epilogue of one tile runs while the tensor core works on its neighbours.
#include <cfloat>

#include "msa_internal.cuh"

namespace msa {
namespace {

// Warp roles: 0-7 softmax epilogue (two warpgroups), 8-11 dQ drain, 12 TMA
// producer, 13 MMA issuer, 14-15 idle.  Register budgets per warpgroup:
// 2 x 128 x 168 + 128 x 96 + 128 x 80 = 65536 = 512 threads x 128 at launch.
constexpr int kBwdThreads = 512;
constexpr int kProducerWarp = 12, kMmaWarp = 13;
constexpr uint32_t kRegsSoftmax = 168, kRegsDq = 96, kRegsCtl = 80;
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
  static constexpr int kDS = 2 * 16384;           // dS^T hi and lo, [128 keys][64 rows] bf16
  static constexpr int kQO = 2 * kQT;             // Q/dO ring stage (freed by the MMAs)
  static constexpr int kMeta = TPT * kQpRow + TPT * kRec;  // q_p rows + records
  static constexpr int kMetaAl = (kMeta + 127) / 128 * 128;
  static constexpr int kFixed = 2 * kKV + kDS;  // K, V, the dS^T buffer
  static constexpr int kBars = 256;
  static constexpr int kRoom = 232448 - 1024 - kFixed - kBars;
  static constexpr int kNQ = (kRoom - 2 * kMetaAl) / kQO < 4 ? (kRoom - 2 * kMetaAl) / kQO : 4;
  static constexpr int kNM = (kRoom - kNQ * kQO) / kMetaAl < 4 ? (kRoom - kNQ * kQO) / kMetaAl : 4;
  static constexpr int kSmem = 1024 + kFixed + kNQ * kQO + kNM * kMetaAl + kBars;
  static_assert(kNQ >= 2 && kNM >= 2, "at least two stages of each ring");
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
  const uint16_t* q;   // [T][hq][d] bf16
  const uint16_t* dO;  // [T][hq][d] bf16
  int chunk;           // query chunk (qchunk_of); >= 0: dK, dV, dk_p accumulate
  int qcb;             // KV blocks per query chunk
};

// acc[k] += v for a warp-uniform runtime k in [0, 32): a switch keeps every
// accumulator in a register.
__device__ __forceinline__ void add_at32(float (&acc)[32], int k, float v) {
  switch (k) {
#define MSA_ADD_CASE(x) \
  case x:               \
    acc[x] += v;        \
    break;
    MSA_ADD_CASE(0) MSA_ADD_CASE(1) MSA_ADD_CASE(2) MSA_ADD_CASE(3) MSA_ADD_CASE(4)
    MSA_ADD_CASE(5) MSA_ADD_CASE(6) MSA_ADD_CASE(7) MSA_ADD_CASE(8) MSA_ADD_CASE(9)
    MSA_ADD_CASE(10) MSA_ADD_CASE(11) MSA_ADD_CASE(12) MSA_ADD_CASE(13) MSA_ADD_CASE(14)
    MSA_ADD_CASE(15) MSA_ADD_CASE(16) MSA_ADD_CASE(17) MSA_ADD_CASE(18) MSA_ADD_CASE(19)
    MSA_ADD_CASE(20) MSA_ADD_CASE(21) MSA_ADD_CASE(22) MSA_ADD_CASE(23) MSA_ADD_CASE(24)
    MSA_ADD_CASE(25) MSA_ADD_CASE(26) MSA_ADD_CASE(27) MSA_ADD_CASE(28) MSA_ADD_CASE(29)
    MSA_ADD_CASE(30) MSA_ADD_CASE(31)
#undef MSA_ADD_CASE
    default:
      break;
  }
}

// Work item of CTA `x`: KV group g, global block gb, the block's token range
// and its list (diagonal tokens first, then the gathered entries).
struct Item {
  int g, gb, j, kstart, nkeys, lbeg, lcnt, ndiag, ntiles, slot_diag;
  int lo;         // first list entry of this launch's query chunk, relative to lbeg
  int t0;         // first token of the query chunk (partial rows are token - t0)
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
  const int lend = a.row_ptr[it.g * a.nb_bound + it.gb + 1];
  // this launch's query chunk: the block's own queries if the block is in it,
  // and the part of its token-sorted list that falls in [t0, t1)
  const QChunk qc = qchunk_of(a.cu, a.cu_blocks, a.ndoc, a.T, nbt, a.chunk, a.qcb);
  int lo = it.lbeg, hi = lend;
  if (a.chunk >= 0) {
    lo = lower_bound_token(a.ent, it.lbeg, lend, qc.t0);
    hi = lower_bound_token(a.ent, lo, lend, qc.t1);
  }
  it.lo = lo - it.lbeg;
  it.lcnt = hi - lo;
  it.t0 = qc.t0;
  it.ndiag = (it.gb >= qc.b0 && it.gb < qc.b1) ? (it.nkeys + TPT - 1) / TPT : 0;
  it.ntiles = it.ndiag + (it.lcnt + TPT - 1) / TPT;
  it.slot_diag = min(it.j, a.K - 1);
  // Records of group g follow those of groups < g (their lists plus T diagonal
  // entries each); inside the group, block gb's diagonal entries are preceded
  // by kstart diagonal entries of earlier blocks.
  it.ext = (long long)it.lbeg + (long long)it.g * a.T + it.kstart;
  return it.ntiles > 0;
}

// First list entry and entry count of tile n.
__device__ __forceinline__ void tile_span(const Item& it, int n, int TPT, int& x0, int& cnt) {
  if (n < it.ndiag) {
    x0 = n * TPT;
    cnt = min(TPT, it.nkeys - x0);
  } else {
    const int m = (n - it.ndiag) * TPT;
    x0 = it.nkeys + it.lo + m;
    cnt = min(TPT, it.lcnt - m);
  }
}

// One record per list entry of every work item, in list order:
//   int {t, slot, arg, g_b bits} then G x float {-LSE log2(e), -scale D},
// padded to 16 bytes (the epilogue then needs one FMA for each exponent and
// one for dP - D).  Entries with an out-of-range token are written with t = T
// and -LSE log2(e) = -inf (the kernel then treats them as padding).
template <int G>
__global__ void __launch_bounds__(128) k_bwd_prep(const BwdArgs a) {
  constexpr int kRec = bwd_rec_bytes(G);
  Item it;
  if (!item_of(blockIdx.x, kRT / G, a, it)) return;
  const int ndg = it.ndiag > 0 ? it.nkeys : 0;  // the block's own queries, if in the chunk
  const int n_ext = ndg + it.lcnt;
  const float gscale = a.kl_weight * a.proxy_scale;
  for (int y = threadIdx.x; y < n_ext; y += blockDim.x) {
    int t, slot, x;
    if (y < ndg) {
      x = y;
      t = it.kstart + x;
      slot = it.slot_diag;
    } else {
      x = it.nkeys + it.lo + (y - ndg);
      const uint32_t e = __ldg(a.ent + it.lbeg + it.lo + (y - ndg));
      t = (int)(e >> 4);
      slot = (int)(e & 15u);
    }
    int4 hdr = make_int4(a.T, 0, 0, 0);
    float2 rows[G];
#pragma unroll
    for (int h = 0; h < G; ++h) rows[h] = make_float2(__int_as_float(0xff800000), 0.f);
    if (t >= 0 && t < a.T) {
      const size_t e = ((size_t)t * a.hkv + it.g) * a.K + slot;
      const float p = __expf(__ldg(a.sel_score + e) - __ldg(a.plse + (size_t)t * a.hkv + it.g));
      const float gs = gscale * (p - __ldg(a.mass + e));
      hdr = make_int4(t, slot, __ldg(a.sel_arg + e) & (kBlock - 1), __float_as_int(gs));
      const size_t r0 = (size_t)t * a.hq + it.g * G;
#pragma unroll
      for (int h = 0; h < G; ++h)
        rows[h] = make_float2(-__ldg(a.lse + r0 + h) * kLog2eB, -a.scale * __ldg(a.dsum + r0 + h));
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
    k_bwd(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
          const __grid_constant__ CUtensorMap tm_qp, const BwdArgs a) {
  using C = BwdCfg<D, G, DP>;
  constexpr int TPT = C::TPT, TPL = C::TPL, NQ = C::kNQ, NM = C::kNM, NCH = D / 64;
  constexpr int kQT = C::kQT, kQChunk = C::kQChunk, kRec = C::kRec;
  // TMEM: slot b (b = tile parity) at columns 128b: [0, 64) S^T, later dQ^T;
  // [64, 128) dP^T, later P^T (bf16 pairs) in the first 16 columns of each
  // warpgroup's half.  dV and dK accumulate over the whole block.
  constexpr uint32_t T_DV = 256, T_DK = 256 + D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + C::kKV;
  uint8_t* sDS = sV + C::kKV;  // {dS^T hi, dS^T lo}, 128B swizzle
  uint8_t* sQO = sDS + C::kDS;
  uint8_t* sMeta = sQO + NQ * C::kQO;
  auto stQ = [&](int s) { return sQO + s * C::kQO; };
  auto stO = [&](int s) { return stQ(s) + kQT; };
  auto stP = [&](int s) { return sMeta + s * C::kMetaAl; };      // q_p rows
  auto stR = [&](int s) { return stP(s) + TPT * C::kQpRow; };   // records
  uint64_t* bars = reinterpret_cast<uint64_t*>(sMeta + NM * C::kMetaAl);
  // Q/dO ring: full (TMA), free (the MMA commit of dV/dK/dQ); metadata ring:
  // full (TMA), free (the softmax and dQ warps).  Per TMEM slot: S^T/dP^T
  // ready, dS^T/P^T ready, dQ^T ready, slot released by the dQ warps.
  const int B_QF = 0, B_QE = NQ, B_MF = 2 * NQ, B_ME = 2 * NQ + NM, B_SP = 2 * NQ + 2 * NM,
            B_DS = B_SP + 2, B_DQ = B_SP + 4, B_SF = B_SP + 6, B_KV = B_SP + 8, B_END = B_SP + 9;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + B_END + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  Item it;
  if (!item_of(blockIdx.x, TPT, a, it)) return;
  const int g = it.g;
  const uint8_t* recg = a.rec + (size_t)it.ext * kRec;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NQ; ++s) {
      mbar_init(bar(B_QF + s), 32);  // one cp.async arrival per producer lane
      mbar_init(bar(B_QE + s), 1);
    }
    for (int s = 0; s < NM; ++s) {
      mbar_init(bar(B_MF + s), 1);
      mbar_init(bar(B_ME + s), 12);  // eight softmax warps and four dQ warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_SP + b), 1);
      mbar_init(bar(B_DS + b), 8);
      mbar_init(bar(B_DQ + b), 1);
      mbar_init(bar(B_SF + b), 4);
    }
    mbar_init(bar(B_KV), 1);
    mbar_init(bar(B_END), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tslot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(tslot);

  if (warp >= 12) {
    setmaxnreg_dec<kRegsCtl>();
    if (warp == kProducerWarp) {
      // ------------------------------ TMA producer ------------------------------
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_KV), 2 * C::kKV);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          tma_load_3d(smem_u32(sK + c * 16384), &tm_k, bar(B_KV), 64 * c, g, it.kstart);
          tma_load_3d(smem_u32(sV + c * 16384), &tm_v, bar(B_KV), 64 * c, g, it.kstart);
        }
      }
      // tokens of the next tile are read one tile ahead (records hold them)
      auto load_tokens = [&](int n, int (&tok)[TPL]) {
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
      int tok[TPL];
      if (it.ntiles > 0) load_tokens(0, tok);
      int issued = 0, missued = 0;  // tiles whose Q/dO, metadata copies were issued
      for (int n = 0; n < it.ntiles; ++n) {
        const int sq = n % NQ, sm = n % NM;
        if (n >= NM && !wait_bar_warp(bar(B_ME + sm), ((n / NM) & 1) ^ 1, abort_flag, a.status,
                                      wait_site(kKerBwd, B_ME + sm, n)))
          break;
        int x0, cnt;
        tile_span(it, n, TPT, x0, cnt);
        missued = n + 1;
        // metadata first: it does not wait for the tensor core
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_MF + sm), TPT * DP * 2 + TPT * kRec);
          bulk_load(smem_u32(stR(sm)), recg + (size_t)x0 * kRec, TPT * kRec, bar(B_MF + sm));
        }
        __syncwarp();
        const uint32_t pb = smem_u32(stP(sm));
#pragma unroll
        for (int u = 0; u < TPL; ++u) {
          const int i = lane + 32 * u;
          if (i < TPT) tma_load_3d(pb + i * C::kQpRow, &tm_qp, bar(B_MF + sm), 0, g, tok[u]);
        }
        if (n >= NQ && !wait_bar_warp(bar(B_QE + sq), ((n / NQ) & 1) ^ 1, abort_flag, a.status,
                                      wait_site(kKerBwd, B_QE + sq, n)))
          break;
        issued = n + 1;
        // Q and dO rows: 16-byte cp.async copies, lanes along a row (coalesced),
        // written in the 128B-swizzled K-major layout the MMAs read; padding
        // rows (token T) are zero-filled.  Each lane arrives on the stage's
        // barrier once its copies have landed.
        {
          constexpr int CPR = D / 8;     // 16-byte chunks per row
          constexpr int RPI = 32 / CPR;  // rows per warp-wide step
          const uint32_t qb = smem_u32(stQ(sq)), ob = smem_u32(stO(sq));
          const int c = lane % CPR;
          const uint32_t cofs = (uint32_t)(c >> 3) * kQChunk;
#pragma unroll 4
          for (int k = 0; k < kRT / RPI; ++k) {
            const int row = RPI * k + lane / CPR;
            const int ti = row / G, h = row % G;
            const int tu = (TPL == 1 || ti < 32) ? tok[0] : tok[TPL - 1];
            const int t = __shfl_sync(0xffffffffu, tu, ti & 31);
            const bool ok = t < a.T;
            const size_t src = ((size_t)(ok ? t : 0) * a.hq + g * G + h) * D + c * 8;
            const uint32_t dst = cofs + (uint32_t)row * 128u + ((((uint32_t)c & 7u) ^ ((uint32_t)row & 7u)) << 4);
            cp_async16(qb + dst, a.q + src, ok ? 16u : 0u);
            cp_async16(ob + dst, a.dO + src, ok ? 16u : 0u);
          }
          cp_async_mbar_arrive(bar(B_QF + sq));
        }
        if (n + 1 < it.ntiles) load_tokens(n + 1, tok);
      }
      // Let this CTA's own copies land before it exits (they have, unless a
      // wait above gave up).
      if (lane == 0) {
        drain_bar(bar(B_KV), 0);
        for (int n = missued > NM ? missued - NM : 0; n < missued; ++n)
          drain_bar(bar(B_MF + n % NM), (n / NM) & 1);
        for (int n = issued > NQ ? issued - NQ : 0; n < issued; ++n)
          drain_bar(bar(B_QF + n % NQ), (n / NQ) & 1);
      }
    } else if (warp == kMmaWarp) {
      // ------------------------------ MMA issuer -------------------------------
      // Order: S^T/dP^T of tile n, then dV/dK/dQ^T of tile n-1.
      if (lane == 0) {
        constexpr uint32_t idST = make_idesc_bf16(128, kRT, false, false);
        constexpr uint32_t idDV = make_idesc_bf16(128, D, false, true);
        constexpr uint32_t idDQ = make_idesc_bf16(128, kRT, true, true);
        bool ok = wait_bar(bar(B_KV), 0, abort_flag, a.status, wait_site(kKerBwd, B_KV, 0));
        const uint32_t k0 = smem_u32(sK), v0 = smem_u32(sV);
        for (int n = 0; ok && n <= it.ntiles; ++n) {
          if (n < it.ntiles) {
            const int s = n % NQ, b = n & 1;
            if (!wait_bar(bar(B_QF + s), (n / NQ) & 1, abort_flag, a.status,
                          wait_site(kKerBwd, B_QF + s, n)))
              break;
            if (n >= 2 && !wait_bar(bar(B_SF + b), ((n >> 1) - 1) & 1, abort_flag, a.status,
                                    wait_site(kKerBwd, B_SF + b, n)))
              break;
            // the Q/dO rows were written by cp.async (generic proxy)
            fence_async_smem();
            tc_fence_after();
            const uint32_t q0 = smem_u32(stQ(s)), o0 = smem_u32(stO(s));
            const uint32_t ts = tbase + 128u * b;
            // S^T = K Q^T and dP^T = V dO^T   (M = 128 keys, N = 64 rows, K = D)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t kv_off = (kk >> 2) * 16384 + (kk & 3) * 32;
              const uint32_t q_off = (kk >> 2) * kQChunk + (kk & 3) * 32;
              umma_bf16(ts, make_sdesc(k0 + kv_off, 16, 1024, kLayoutSW128),
                        make_sdesc(q0 + q_off, 16, 1024, kLayoutSW128), idST, kk > 0);
              umma_bf16(ts + 64, make_sdesc(v0 + kv_off, 16, 1024, kLayoutSW128),
                        make_sdesc(o0 + q_off, 16, 1024, kLayoutSW128), idST, kk > 0);
            }
            umma_commit(bar(B_SP + b));
          }
          if (n >= 1) {
            const int m = n - 1, s = m % NQ, b = m & 1;
            if (!wait_bar(bar(B_DS + b), (m >> 1) & 1, abort_flag, a.status,
                          wait_site(kKerBwd, B_DS + b, m)))
              break;
            tc_fence_after();
            const uint32_t q0 = smem_u32(stQ(s)), o0 = smem_u32(stO(s));
            const uint32_t ds0 = smem_u32(sDS), dl0 = ds0 + 16384;
            const uint32_t ts = tbase + 128u * b;
            // dV += P^T dO (P^T from TMEM), dK += (dS_hi + dS_lo)^T Q
            // (M = 128 keys, N = D, K = 64 rows)
#pragma unroll
            for (int kk = 0; kk < kRT / 16; ++kk) {
              const uint32_t acc = (m > 0 || kk > 0) ? 1u : 0u;
              const uint64_t bdo = make_sdesc(o0 + kk * 2048, kQChunk, 1024, kLayoutSW128);
              const uint64_t bq = make_sdesc(q0 + kk * 2048, kQChunk, 1024, kLayoutSW128);
              umma_bf16_ts(tbase + T_DV, ts + 64 + 32 * (kk >> 1) + 8 * (kk & 1), bdo, idDV, acc);
              umma_bf16(tbase + T_DK, make_sdesc(ds0 + kk * 32, 16, 1024, kLayoutSW128), bq,
                        idDV, acc);
              umma_bf16(tbase + T_DK, make_sdesc(dl0 + kk * 32, 16, 1024, kLayoutSW128), bq,
                        idDV, 1u);
            }
            // dQ^T = K^T (dS_hi + dS_lo)^T into the slot's S^T columns
            // (M = D padded to 128, N = 64 rows, K = 128 keys)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t ak = make_sdesc(k0 + kk * 2048, 16384, 1024, kLayoutSW128);
              umma_bf16(ts, ak, make_sdesc(ds0 + kk * 2048, 16384, 1024, kLayoutSW128), idDQ,
                        kk > 0);
              umma_bf16(ts, ak, make_sdesc(dl0 + kk * 2048, 16384, 1024, kLayoutSW128), idDQ,
                        1u);
            }
            umma_commit(bar(B_DQ + b));
            umma_commit(bar(B_QE + s));
          }
        }
        // every MMA issued by this CTA completes before TMEM is released
        umma_commit(bar(B_END));
        drain_bar(bar(B_END), 0);
      }
    }
  } else if (warp >= 8) {
    setmaxnreg_dec<kRegsDq>();
    // ------------------------------ dQ drain -----------------------------------
    // Warp w reads TMEM lanes 32(w-8).. (head-dim index kk) of the slot's dQ^T
    // (64 row columns), releases the slot to the MMA warp, then writes the
    // dq_part rows: one coalesced 128-byte store per warp and row.
    const int kk = (warp - 8) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp - 8) * 32) << 16;
    bool dead = false;
    for (int m = 0; m < it.ntiles; ++m) {
      const int s = m % NM, b = m & 1;
      dead = dead || !wait_bar_warp(bar(B_MF + s), (m / NM) & 1, abort_flag, a.status,
                                    wait_site(kKerBwd, B_MF + s, m));
      dead = dead || !wait_bar_warp(bar(B_DQ + b), (m >> 1) & 1, abort_flag, a.status,
                                    wait_site(kKerBwd, B_DQ + b, m));
      tc_fence_after();
      const bool act = !dead && (warp - 8) * 32 < D;  // warp-uniform
      uint32_t va[32], vb[32];  // rows 0..31 and 32..63 of the tile
      if (act) tmem_ld32x2(tbase + lane_off + 128u * b, tbase + lane_off + 128u * b + 32, va, vb);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SF + b));
      if (act) {
        int x0, cnt;
        tile_span(it, m, TPT, x0, cnt);
        const uint8_t* rec = stR(s);
#pragma unroll
        for (int ti = 0; ti < TPT; ++ti) {
          if (ti < cnt) {
            const int4 hd = *reinterpret_cast<const int4*>(rec + ti * kRec);
            if (hd.x < a.T) {
              float* dst = a.dq_part +
                           (((size_t)(hd.x - it.t0) * a.hq + g * G) * a.K + hd.y) * (size_t)D + kk;
#pragma unroll
              for (int h = 0; h < G; ++h) {
                const int r = ti * G + h;
                dst[(size_t)h * a.K * D] = __uint_as_float(r < 32 ? va[r] : vb[r - 32]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_ME + s));
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------ softmax epilogue ----------------------------
    // Two warpgroups: warpgroup e owns tile rows 32e..32e+31 (columns of S^T
    // and dP^T) for all 128 keys.  Abort-safe: a failed wait marks the warp
    // dead; it still walks every tile and arrives on every barrier.
    const int e = warp >> 2;
    const int kk = (warp & 3) * 32 + lane;  // key: TMEM lane of S^T, dP^T, dV, dK
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale * kLog2eB;
    // Proxy key gradient: lane l of warpgroup e holds dimension DPH e + l of
    // dk_p for the warp's 32 keys (kacc[k] <-> key 32 (warp & 3) + k).
    constexpr int DPH = DP / 2;
    float kacc[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) kacc[k] = 0.f;
    bool dead = false;
    for (int n = 0; n < it.ntiles; ++n) {
      const int s = n % NM, b = n & 1;
      int x0, cnt;
      tile_span(it, n, TPT, x0, cnt);
      const bool diag = n < it.ndiag;
      const bool masked = diag || cnt < TPT;
      const uint8_t* rec = stR(s);
      uint8_t* dsh = sDS;
      uint8_t* dsl = dsh + 16384;
      dead = dead || !wait_bar_warp(bar(B_MF + s), (n / NM) & 1, abort_flag, a.status,
                                    wait_site(kKerBwd, B_MF + s, n));
      if (!dead) {
        // fused proxy gradient (needs only the tile's records and q_p rows, so
        // it runs while the S^T/dP^T products are in flight): every token of the
        // tile adds g_b q_p[t] to the dk_p row of its block argmax; the warp
        // owning that key takes it, one dimension per lane (tokens in list
        // order, so the sum is deterministic)
        for (int base = 0; base < cnt; base += 32) {
          const int i = base + lane;
          int ai = -1;
          float gi = 0.f;
          if (i < cnt) {
            const int4 hd = *reinterpret_cast<const int4*>(rec + i * kRec);
            if (hd.x < a.T) {
              ai = hd.z;
              gi = __int_as_float(hd.w);
            }
          }
          uint32_t mine = __ballot_sync(0xffffffffu, ai >= 0 && (ai >> 5) == (warp & 3));
          while (mine) {
            const int j = __ffs(mine) - 1;
            mine &= mine - 1;
            const int aj = __shfl_sync(0xffffffffu, ai, j);
            const float gj = __shfl_sync(0xffffffffu, gi, j);
            const float qv =
                lane < DPH ? __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(
                                                 stP(s) + (base + j) * C::kQpRow +
                                                 (DPH * e + lane) * 2)
                                             << 16)
                           : 0.f;
            add_at32(kacc, aj & 31, gj * qv);
          }
        }
      }
      dead = dead || !wait_bar_warp(bar(B_SP + b), (n >> 1) & 1, abort_flag, a.status,
                                    wait_site(kKerBwd, B_SP + b, n));
      tc_fence_after();
      if (!dead) {
        const uint32_t ts = tbase + lane_off + 128u * b;
        // P^T and dS^T of this warpgroup's 32 rows (bf16 pairs); the dS^T
        // stores are the only step that waits for the previous tile's products
        uint32_t pw[16], dh[16], dl[16];
        // this warpgroup's rows start at token 32e/G of the tile; every offset
        // below is a compile-time constant
        const uint8_t* recw = rec + (32 * e / G) * kRec + 16;
        const int tw0 = 32 * e / G;
#pragma unroll
        for (int q16 = 0; q16 < 2; ++q16) {
          const int r0 = 32 * e + 16 * q16;
          uint32_t sv[16], dv[16];
          tmem_ld16x2(ts + r0, ts + 64 + r0, sv, dv);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float pv[2];
            uint32_t hb[2], lb[2];
            // rows 2i, 2i+1 of the half: record entries {-LSE log2(e), -scale D}
            float2 ldp[2];
            const int rl = 16 * q16 + 2 * i;
            if (G >= 2) {  // the two rows are heads h, h+1 of one token
              const float4 x = *reinterpret_cast<const float4*>(recw + (rl / G) * kRec + 8 * (rl % G));
              ldp[0] = make_float2(x.x, x.y);
              ldp[1] = make_float2(x.z, x.w);
            } else {
              ldp[0] = *reinterpret_cast<const float2*>(recw + rl * kRec);
              ldp[1] = *reinterpret_cast<const float2*>(recw + (rl + 1) * kRec);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int ti = tw0 + (rl + u) / G;
              const float2 ld = ldp[u];
              float p = ex2_approx(fmaf(__uint_as_float(sv[2 * i + u]), sl2, ld.x));
              float ds = p * fmaf(__uint_as_float(dv[2 * i + u]), a.scale, ld.y);
              if (masked) {
                const bool use = ti < cnt && (!diag || kk <= x0 + ti);
                p = use ? p : 0.f;
                ds = use ? ds : 0.f;
              }
              pv[u] = p;
              // dS = hi + lo with hi its bf16 truncation (exact split in fp32);
              // lo is truncated to bf16 as well: |error| < 2^-15 |dS|.
              hb[u] = __float_as_uint(ds);
              lb[u] = __float_as_uint(ds - __uint_as_float(hb[u] & 0xFFFF0000u));
            }
            pw[8 * q16 + i] = pack_bf16(pv[0], pv[1]);
            dh[8 * q16 + i] = pack_hi_halves(hb[0], hb[1]);
            dl[8 * q16 + i] = pack_hi_halves(lb[0], lb[1]);
          }
        }
        // P^T into this warpgroup's half of the dP^T columns (already read)
        tmem_st16(ts + 64 + 32 * e, pw);
        // the dS^T buffer was last read by the products of tile n-1
        if (n >= 1)
          dead = !wait_bar_warp(bar(B_DQ + ((n - 1) & 1)), ((n - 1) >> 1) & 1, abort_flag,
                                a.status, wait_site(kKerBwd, B_DQ + ((n - 1) & 1), n));
        if (!dead) {
#pragma unroll
          for (int q16 = 0; q16 < 2; ++q16) {
            const int r0 = 32 * e + 16 * q16;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const uint32_t off = sw128_offset((uint32_t)kk, (uint32_t)(r0 / 8 + q));
              const int w0 = 8 * q16 + 4 * q;
              *reinterpret_cast<uint4*>(dsh + off) =
                  make_uint4(dh[w0], dh[w0 + 1], dh[w0 + 2], dh[w0 + 3]);
              *reinterpret_cast<uint4*>(dsl + off) =
                  make_uint4(dl[w0], dl[w0 + 1], dl[w0 + 2], dl[w0 + 3]);
            }
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_DS + b));
        mbar_arrive(bar(B_ME + s));
      }
    }

    // dK, dV and dk_p rows of this block (lane = key), written once after the
    // last products have completed.  Warpgroup 0 writes dV, warpgroup 1 dK,
    // each its half of dk_p.  The TMEM loads are warp-collective, so every lane
    // executes them; only the stores depend on the key being inside the
    // document.
    if (it.ntiles > 0) {
      const int m = it.ntiles - 1;
      dead = dead || !wait_bar_warp(bar(B_DQ + (m & 1)), (m >> 1) & 1, abort_flag, a.status,
                                    wait_site(kKerBwd, B_DQ + (m & 1), m));
    }
    tc_fence_after();
    if (!dead) {
      // dk_p first: its 32 accumulators are dead before the TMEM reads below
      if (lane < DPH) {
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int key = (warp & 3) * 32 + k;
          if (key < it.nkeys) {
            float* pk = a.dk_p + ((size_t)(it.kstart + key) * a.hkv + g) * DP + DPH * e + lane;
            *pk = a.chunk >= 0 ? *pk + kacc[k] : kacc[k];
          }
        }
      }
      const bool keep = kk < it.nkeys;
      const size_t krow = (size_t)(it.kstart + (keep ? kk : 0)) * a.hkv + g;
      float* outr = (e == 0 ? a.dv : a.dk) + krow * D;
      const uint32_t tcol = e == 0 ? T_DV : T_DK;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32f(tbase + lane_off + tcol + c * 32, v);
        if (keep) {
          float4* o4 = reinterpret_cast<float4*>(outr + c * 32);
          if (a.chunk < 0) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              o4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          } else {
            // query chunks add up, in chunk order; one float4 at a time (the
            // empty asm keeps the loads from being batched up front)
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 y = o4[q];
              o4[q] = make_float4(y.x + v[4 * q], y.y + v[4 * q + 1], y.z + v[4 * q + 2],
                                  y.w + v[4 * q + 3]);
              asm volatile("" ::: "memory");
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
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
  // The warpgroups' register budgets are drawn from the registers the block
  // is launched with; a larger sum would leave setmaxnreg.inc waiting.
  constexpr int kBudget = 2 * 128 * kRegsSoftmax + 128 * kRegsDq + 128 * kRegsCtl;
  static_assert(kBudget <= 65536, "register budgets exceed the register file");
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, k_bwd<D, G, DP>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kBwdThreads < kBudget) return cudaErrorInvalidConfiguration;
  k_bwd_prep<G><<<s.nb_bound * s.hkv, 128, 0, st>>>(a);
  e = cudaFuncSetAttribute(k_bwd<D, G, DP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmem);
  if (e != cudaSuccess) return e;
  k_bwd<D, G, DP><<<s.nb_bound * s.hkv, kBwdThreads, C::kSmem, st>>>(m[0], m[1], m[2], a);
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
                       float* dv, float* dk_p, int chunk, unsigned* status, cudaStream_t st) {
  // K, V and q_p rows by TMA; Q and dO rows are gathered by cp.async in the kernel
  CUtensorMap m[3];
  cudaError_t e;
  if ((e = make_tmap_3d(&m[0], k, s.d, s.hkv, s.T, 64, 1, 128, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&m[1], v, s.d, s.hkv, s.T, 64, 1, 128, 128)) != cudaSuccess) return e;
  if ((e = make_tmap_3d(&m[2], q_p, s.dp, s.hkv, s.T, s.dp, 1, 1, 0)) != cudaSuccess) return e;
  BwdArgs a{cu_seqlens, cu_blocks, row_ptr,    ent,        rec,          lse,         dsum,
            mass,       sel_score, sel_arg,    plse,       s.ndoc,       s.T,         s.hq,
            s.hkv,      s.K,       s.nb_bound, s.softmax_scale, s.proxy_scale, s.kl_weight,
            dq_part,    dk,        dv,         dk_p,       status,       q,           dO,
            chunk,      s.qc_blocks};
  if (s.d == 128)
    return s.dp == 64 ? launch_bwd_g<128, 64>(s, m, a, st) : launch_bwd_g<128, 32>(s, m, a, st);
  return s.dp == 64 ? launch_bwd_g<64, 64>(s, m, a, st) : launch_bwd_g<64, 32>(s, m, a, st);
}

}  // namespace msa
