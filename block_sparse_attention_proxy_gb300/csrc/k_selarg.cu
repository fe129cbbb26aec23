// Block argmax of the proxy scores for every (token, selected earlier block).
//
// The proxy picks KV blocks by the maximum proxy score inside each 128-key
// block ("Dramatically Speeding Up Million-Token Training! ... 'Flash-MSA'
// ...", ai-minor.com, "What's Happening? News Overview"); the gradient of the
// proxy loss reaches k_p through the key attaining that maximum.  The
// selector keeps only the block maxima while it streams over all earlier
// blocks (and the argmax of the diagonal block); the argmax of each of the
// k - 1 chosen earlier blocks is found here, KV-major, from the regrouped
// lists (the queries that chose each block), so it costs one score tile per
// 128 choosers instead of bookkeeping on every (query, block) pair.
//
// One CTA of 128 threads per (KV group g, KV block b): the block's k_p rows
// are loaded once by TMA; per tile of 128 choosers their q_p rows are
// gathered with cp.async into the swizzled K-major layout, one MMA chain
// (M = 128 choosers, N = 128 keys, K = dp) computes the scores into TMEM, and
// thread r (TMEM lane r) takes the lowest key attaining its row maximum.
#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kArgThreads = 128;

struct ArgArgs {
  const int32_t* cu;
  const int32_t* cu_blocks;
  const int32_t* row_ptr;
  const uint32_t* ent;
  const uint16_t* q_p;
  int ndoc, T, hkv, K, nb_bound;
  uint8_t* sel_arg;
  unsigned* status;
};

// Maximum of 32 scores held as raw fp32 bits, and the lowest index attaining it.
__device__ __forceinline__ float max32_of(const uint32_t (&r)[32]) {
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
__device__ __forceinline__ int first_eq32(const uint32_t (&r)[32], float v) {
  int a = 32;
#pragma unroll
  for (int i = 31; i >= 0; --i) a = (__uint_as_float(r[i]) == v) ? i : a;
  return a;
}

template <int DP>
__global__ void __launch_bounds__(kArgThreads)
    k_sel_arg(const __grid_constant__ CUtensorMap tm_kp, const ArgArgs a) {
  constexpr int kRow = DP * 2;  // bytes of one q_p / k_p row
  constexpr int kTile = 128 * kRow;
  constexpr uint32_t kLayout = DP == 64 ? kLayoutSW128 : kLayoutSW64;
  constexpr uint32_t kSBO = 8 * kRow;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;          // k_p block, 128 keys
  uint8_t* sQ = sK + kTile;    // q_p rows of the current 128 choosers
  uint64_t* bars = reinterpret_cast<uint64_t*>(sQ + kTile);  // 0 k_p loaded, 1 scores ready
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  const int tid = threadIdx.x, warp = tid >> 5;

  if (!a.cu_blocks[a.ndoc + 1]) return;  // malformed cu_seqlens (flagged by k_meta)
  const int nbt = min(a.cu_blocks[a.ndoc], a.nb_bound);
  const int g = blockIdx.x % a.hkv;
  const int gb = (int)(blockIdx.x / a.hkv);
  if (gb >= nbt) return;
  const int lbeg = a.row_ptr[g * a.nb_bound + gb];
  const int lcnt = a.row_ptr[g * a.nb_bound + gb + 1] - lbeg;
  if (lcnt <= 0) return;
  const int d = doc_of_block(a.cu_blocks, a.ndoc, gb);
  const int kstart = a.cu[d] + (gb - a.cu_blocks[d]) * kBlock;

  const uint32_t b_kp = smem_u32(bars), b_mma = smem_u32(bars + 1);
  if (tid == 0) {
    mbar_init(b_kp, 1);
    mbar_init(b_mma, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(tslot);
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

  if (tid == 0) {
    mbar_arrive_expect_tx(b_kp, kTile);
    tma_load_3d(smem_u32(sK), &tm_kp, b_kp, 0, g, kstart);
  }
  // A gathered block lies wholly before its chooser's own block, so all 128
  // keys are real keys of the document.
  bool dead = !wait_bar_warp(b_kp, 0, abort_flag, a.status, wait_site(kKerSelArg, 0, 0));
  int issued = 0;
  const int ntile = (lcnt + 127) / 128;
  for (int n = 0; n < ntile; ++n) {
    // thread tid gathers chooser row tid of the tile (zero row past the list)
    const int x = n * 128 + tid;
    int t = a.T, slot = 0;
    if (x < lcnt) {
      const uint32_t e = __ldg(a.ent + lbeg + x);
      t = (int)(e >> 4);
      slot = (int)(e & 15u);
    }
    const bool valid = t < a.T;
    const uint16_t* src = a.q_p + ((size_t)(valid ? t : 0) * a.hkv + g) * DP;
#pragma unroll
    for (int c = 0; c < kRow / 16; ++c) {
      const int pc = DP == 64 ? (c ^ (tid & 7)) : (c ^ ((tid >> 1) & 3));
      cp_async16(smem_u32(sQ + tid * kRow + pc * 16), src + c * 8, valid ? 16u : 0u);
    }
    cp_async_wait_all();
    fence_async_smem();  // generic-proxy writes -> the MMA's reads
    __syncthreads();
    if (tid == 0 && !dead) {
      tc_fence_after();
      constexpr uint32_t idesc = make_idesc_bf16(128, 128, false, false);
      const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK);
#pragma unroll
      for (int kk = 0; kk < DP / 16; ++kk)
        umma_bf16(tbase, make_sdesc(q0 + kk * 32, 16, kSBO, kLayout),
                  make_sdesc(k0 + kk * 32, 16, kSBO, kLayout), idesc, kk > 0);
      umma_commit(b_mma);
      ++issued;
    }
    dead = dead || !wait_bar_warp(b_mma, n & 1, abort_flag, a.status, wait_site(kKerSelArg, 1, n));
    tc_fence_after();
    if (!dead) {
      uint32_t va[32], vb[32], vc[32], vd[32];
      tmem_ld32x2(tbase + lane_off, tbase + lane_off + 32, va, vb);
      tmem_ld32x2(tbase + lane_off + 64, tbase + lane_off + 96, vc, vd);
      const float ma = max32_of(va), mb = max32_of(vb), mc = max32_of(vc), md = max32_of(vd);
      const float best = fmaxf(fmaxf(ma, mb), fmaxf(mc, md));
      int arg;
      if (ma == best)
        arg = first_eq32(va, best);
      else if (mb == best)
        arg = 32 + first_eq32(vb, best);
      else if (mc == best)
        arg = 64 + first_eq32(vc, best);
      else
        arg = 96 + first_eq32(vd, best);
      if (valid) a.sel_arg[((size_t)t * a.hkv + g) * a.K + slot] = (uint8_t)arg;
    }
    tc_fence_before();
    __syncthreads();  // the next tile overwrites sQ and the scores
  }
  if (tid == 0 && issued > 0) drain_bar(b_mma, (issued - 1) & 1);  // set only after an abort
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 128);
  }
}

template <int DP>
cudaError_t launch_sel_arg_t(const Shape& s, const CUtensorMap& mk, const ArgArgs& a,
                             cudaStream_t st) {
  // 56 KB of shared memory keeps at most four CTAs (4 x 128 TMEM columns) per SM
  const size_t smem = 56 * 1024;
  static_assert(1024 + 2 * 128 * DP * 2 + 64 <= 56 * 1024, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(k_sel_arg<DP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  k_sel_arg<DP><<<s.nb_bound * s.hkv, kArgThreads, smem, st>>>(mk, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sel_arg(const Shape& s, const int32_t* cu_seqlens, const int32_t* cu_blocks,
                           const int32_t* row_ptr, const uint32_t* ent, const uint16_t* q_p,
                           const uint16_t* k_p, uint8_t* sel_arg, unsigned* status,
                           cudaStream_t st) {
  CUtensorMap mk;
  const int sw = s.dp == 64 ? 128 : 64;
  cudaError_t e;
  if ((e = make_tmap_3d(&mk, k_p, s.dp, s.hkv, s.T, s.dp, 1, 128, sw)) != cudaSuccess) return e;
  ArgArgs a{cu_seqlens, cu_blocks, row_ptr, ent, q_p, s.ndoc, s.T, s.hkv, s.K, s.nb_bound,
            sel_arg, status};
  return s.dp == 64 ? launch_sel_arg_t<64>(s, mk, a, st) : launch_sel_arg_t<32>(s, mk, a, st);
}

}  // namespace msa
