// Row statistics with the top-p (nucleus) threshold, for temperature > 0 and
// top_p < 1.
//
// Source: "LLM inference acceleration in practice: draft models and
// speculative sampling explained" (mlqm.cn), §4.2 _apply_top_p: rank the
// logits in descending order, keep rank r iff r == 0 or the softmax mass of
// the ranks before it is at most top_p; equal logits are ranked by lower
// index (EAGLE3 draft rows: by target id).
//
// Layout: one row per thread-block cluster of L.cl blocks.  Every thread keeps
// its part of the row in registers for the whole kernel (NV 16-byte vectors),
// so the row is read from HBM exactly once.  The per-element work has no
// atomics:
//   1. row maximum m (block, then cluster through distributed shared memory);
//   2. pass A: e = 2^(l*c - m*c) (c = log2(e)/T) is added to a per-thread
//      private histogram keyed by the exponent and top mantissa bit of e
//      (64 bins, [bin][thread] layout, conflict free).  The cluster adds the
//      bins; the bin b* where the cumulative mass from the top first exceeds
//      top_p * S holds the cut (S = total mass);
//   3. pass B: only elements of bin b* (a few percent of the row) are
//      compacted into a shared list and histogrammed on the next 8 mantissa
//      bits of e with 32-bit atomics; up to three such levels narrow the cut
//      to at most 64 elements, which one warp of the cluster's first block
//      sorts by (logit descending, tie key ascending) and walks exactly.
// Rare rows (the cut in the open bin of tiny masses, a candidate list
// overflow, or more than 64 elements with the same e but different logits)
// take an exact generic radix select over the order keys of all elements.
#include "sv_rows.cuh"

namespace sv {

constexpr int kTpThreads = 256;
constexpr int kNB = 64;            // pass-A bins
constexpr int kCap = 2048;         // candidate list capacity per block
constexpr int kFinal = 64;         // elements resolved by the final sort
constexpr double kScale40 = 1099511627776.0;  // generic path: masses in units of 2^-40
constexpr double kInv40 = 1.0 / 1099511627776.0;

struct TpShared {
  float phist[kNB * kTpThreads];   // [bin][thread] private masses
  float cta_bins[kNB];
  unsigned lvl[2][4][256];         // [buffer][count, mass bits 0-15, 16-31, 32-47][bin]
  unsigned long long tmass[256];
  unsigned tcnt[256];
  uint32_t cbits[kCap];            // candidate logits (float bits)
  int32_t csec[kCap];              // candidate tie keys
  uint32_t gbits[kFinal];          // final group (first block only)
  int32_t gsec[kFinal];
  int gn;
  int cn;
  int flags;
  int wcnt[kTpThreads / 32];
  float red_f[32];
  unsigned long long red_u[32];
  float cta_max;
  uint32_t kmin, kmax;
  int sel;
  int found;   // a bin where the cumulative mass exceeds the limit exists
  unsigned long long sel_above;
  unsigned sel_cnt;
  int bstar;
  double above0;
  double limit;
  double total;
};

// Bin of a mass e in (0, ~1]: 0 for e >= 1.5, then half-octaves downwards;
// e below 2^-30.5 (and 0) land in the open bin kNB-1.
__device__ __forceinline__ int mass_bin(float e) {
  const int b = 255 - static_cast<int>(__float_as_uint(e) >> 22);
  return min(kNB - 1, max(0, b));
}

// exp2 that the compiler may not merge with an earlier identical one: the
// passes after pass A recompute e instead of keeping every e of the row live.
__device__ __forceinline__ float ex2v(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


template <int THREADS>
__device__ __forceinline__ uint32_t block_min_u32(uint32_t v, unsigned long long* scratch) {
  return static_cast<uint32_t>(~block_max_u64<THREADS>(~static_cast<unsigned long long>(v) & 0xffffffffull,
                                                       scratch) & 0xffffffffull);
}

// Sum the three 256-bin level histograms of every block of the cluster.
__device__ __forceinline__ void reduce_levels(cg::cluster_group& cluster, TpShared& sh, int buf, int cl) {
  __syncthreads();
  cluster.sync();
  for (int t = threadIdx.x; t < 256; t += kTpThreads) {
    // All remote loads are issued before any is used (cl <= 16).
    unsigned c[16], l0[16], l1[16], l2[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      if (q < cl) {
        const TpShared* p = cluster.map_shared_rank(&sh, q);
        c[q] = p->lvl[buf][0][t];
        l0[q] = p->lvl[buf][1][t];
        l1[q] = p->lvl[buf][2][t];
        l2[q] = p->lvl[buf][3][t];
      } else {
        c[q] = l0[q] = l1[q] = l2[q] = 0u;
      }
    }
    unsigned long long s0 = 0, s1 = 0, s2 = 0;
    unsigned cnt = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      cnt += c[q];
      s0 += l0[q];
      s1 += l1[q];
      s2 += l2[q];
    }
    sh.tcnt[t] = cnt;
    sh.tmass[t] = s0 + (s1 << 16) + (s2 << 32);
  }
  __syncthreads();
}

// Warp 0: first bin, walking from `top` down to 0, where above + mass > limit.
// If none, the lowest non-empty bin (the cut lies at the end of the range).
__device__ __forceinline__ void level_crossing(TpShared& sh, int top, unsigned long long above,
                                               unsigned long long limit) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  unsigned long long local = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int bin = top - (lane * 8 + k);
    if (bin >= 0) local += sh.tmass[bin];
  }
  unsigned long long incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  unsigned long long run = above + incl - local;
  int hit = -1, last = -1;
  unsigned long long hit_above = 0, last_above = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int bin = top - (lane * 8 + k);
    if (bin < 0) break;
    const unsigned long long ms = sh.tmass[bin];
    if (hit < 0 && run + ms > limit) {
      hit = bin;
      hit_above = run;
    }
    if (sh.tcnt[bin]) {
      last = bin;
      last_above = run;
    }
    run += ms;
  }
  const unsigned hb = __ballot_sync(0xffffffffu, hit >= 0);
  const unsigned lb = __ballot_sync(0xffffffffu, last >= 0);
  int src, b;
  unsigned long long a;
  if (hb) {
    src = __ffs(hb) - 1;
    b = __shfl_sync(0xffffffffu, hit, src);
    a = __shfl_sync(0xffffffffu, hit_above, src);
  } else {
    src = lb ? 31 - __clz(lb) : 0;
    b = __shfl_sync(0xffffffffu, last, src);
    a = __shfl_sync(0xffffffffu, last_above, src);
  }
  if (lane == 0) {
    sh.found = hb != 0;
    sh.sel = b;
    sh.sel_above = a;
    sh.sel_cnt = b >= 0 ? sh.tcnt[b] : 0u;
  }
}

// Warp 0: first bin from 0 upwards where the running count reaches `need`.
__device__ __forceinline__ void count_crossing(TpShared& sh, unsigned need) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  unsigned local = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) local += sh.tcnt[lane * 8 + k];
  unsigned incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  unsigned run = incl - local;
  int hit = -1;
  unsigned before = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const unsigned cnt = sh.tcnt[lane * 8 + k];
    if (hit < 0 && run + cnt >= need) {
      hit = lane * 8 + k;
      before = run;
    }
    run += cnt;
  }
  const unsigned hb = __ballot_sync(0xffffffffu, hit >= 0);
  const int src = hb ? __ffs(hb) - 1 : 31;
  const int b = __shfl_sync(0xffffffffu, hit, src);
  const unsigned bf = __shfl_sync(0xffffffffu, before, src);
  if (lane == 0) {
    sh.sel = b < 0 ? 255 : b;
    sh.sel_above = bf;
  }
}

template <typename E, int NV>
struct RowRegs {
  static constexpr int EPV = Elem<E>::kPerVec;
  uint4 raw[NV];
  float xv;   // extra scalar element (head/tail of an unaligned row), -inf if none
  int xi;     // its index, -1 if none
  int vbase;  // first body vector of this block
  int head;   // elements before the first aligned vector of the row

  // bf16 halves are widened with volatile asm so that the compiler widens
  // them again in every pass instead of keeping all widened values live.
  __device__ __forceinline__ float val(int k, int i) const {
    const uint4& v = raw[k];
    if constexpr (sizeof(E) == 4) {
      return Elem<E>::at(v, i);
    } else {
      const uint32_t w = (i >> 1) == 0 ? v.x : (i >> 1) == 1 ? v.y : (i >> 1) == 2 ? v.z : v.w;
      uint32_t r;
      if (i & 1) asm volatile("and.b32 %0, %1, 0xffff0000;" : "=r"(r) : "r"(w));
      else asm volatile("shl.b32 %0, %1, 16;" : "=r"(r) : "r"(w));
      return __uint_as_float(r);
    }
  }
  __device__ __forceinline__ int idx(int k, int i) const {
    return head + (vbase + k * kTpThreads + static_cast<int>(threadIdx.x)) * EPV + i;
  }
};

template <typename E, int NV>
__device__ __forceinline__ float load_row_regs(RowRegs<E, NV>& R, const E* row, int len, int rank) {
  constexpr int EPV = Elem<E>::kPerVec;
  const RowSplit rs = split_row(row, len);
  R.head = rs.head;
  R.vbase = rank * NV * kTpThreads;
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  float mx = -CUDART_INF_F;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int v = R.vbase + k * kTpThreads + static_cast<int>(threadIdx.x);
    R.raw[k] = v < rs.nvec ? ldg_stream(vp + v) : Elem<E>::neg_inf_vec();
  }
  R.xv = -CUDART_INF_F;
  R.xi = -1;
  if (rank == 0) {
    const int t = threadIdx.x;
    const int ntail = len - rs.tail0;
    if (t < rs.head) R.xi = t;
    else if (t < rs.head + ntail) R.xi = rs.tail0 + (t - rs.head);
    if (R.xi >= 0) R.xv = Elem<E>::load(row + R.xi);
  }
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int i = 0; i < EPV; ++i) mx = fmaxf(mx, R.val(k, i));
  return fmaxf(mx, R.xv);
}

// Exact generic path: radix select over the 32-bit order keys of all
// elements with (count, fixed-point mass) histograms, then the tie cut.  It
// re-reads the block's slice from global memory (it is rare, and this keeps
// the register-resident row out of its live range).  Returns tau, cut and
// the kept mass K (in units of e).
template <typename E, int NV, typename F>
__device__ __forceinline__ void for_slice(const E* row, int len, int rank, F&& f) {
  constexpr int EPV = Elem<E>::kPerVec;
  const RowSplit rs = split_row(row, len);
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  const int vbase = rank * NV * kTpThreads;
#pragma unroll 1
  for (int k = 0; k < NV; ++k) {
    const int v = vbase + k * kTpThreads + static_cast<int>(threadIdx.x);
    if (v >= rs.nvec) break;
    const uint4 w = ldg_stream(vp + v);
#pragma unroll
    for (int i = 0; i < EPV; ++i) f(Elem<E>::at(w, i), rs.head + v * EPV + i);
  }
  if (rank == 0) {
    const int t = threadIdx.x;
    const int ntail = len - rs.tail0;
    int j = -1;
    if (t < rs.head) j = t;
    else if (t < rs.head + ntail) j = rs.tail0 + (t - rs.head);
    if (j >= 0) f(Elem<E>::load(row + j), j);
  }
}

template <typename E, int NV>
__device__ __noinline__ void generic_select(cg::cluster_group& cluster, TpShared& sh, const E* row,
                                            const RowSet& S, int rank, int cl, float c, float mc, float top_p,
                                            int pass_no, uint32_t& tau_out, int32_t& cut_out, double& K_out) {
  constexpr int kPasses = sizeof(E) == 2 ? 2 : 4;
  uint32_t prefix = 0;
  unsigned long long above = 0, limit = 0, total = 0, grp_mass = 0;
  unsigned grp_cnt = 0;
  bool keep_all = false;
#pragma unroll 1
  for (int p = 0; p < kPasses; ++p, ++pass_no) {
    const int buf = pass_no & 1;
    const int sb = 24 - 8 * p;
    for (int t = threadIdx.x; t < 4 * 256; t += kTpThreads) (&sh.lvl[buf][0][0])[t] = 0u;
    __syncthreads();
    for_slice<E, NV>(row, S.len, rank, [&](float x, int) {
      const uint32_t key = order_key(x);
      if (p == 0 || (key >> (sb + 8)) == prefix) {
        const int bin = (key >> sb) & 255;
        // 40-bit fixed point (e <= ~1): exact sums for a whole row.
        const unsigned long long v = __double2ull_rn(static_cast<double>(ex2v(fmaf(x, c, -mc))) * kScale40);
        atomicAdd(&sh.lvl[buf][0][bin], 1u);
        if (v) {
          atomicAdd(&sh.lvl[buf][1][bin], static_cast<unsigned>(v & 0xffffu));
          atomicAdd(&sh.lvl[buf][2][bin], static_cast<unsigned>((v >> 16) & 0xffffu));
          atomicAdd(&sh.lvl[buf][3][bin], static_cast<unsigned>(v >> 32));
        }
      }
    });
    reduce_levels(cluster, sh, buf, cl);
    if (p == 0) {
      unsigned long long part = 0;
      for (int t = threadIdx.x; t < 256; t += kTpThreads) part += sh.tmass[t];
      total = block_sum_u64<kTpThreads>(part, sh.red_u);
      limit = static_cast<unsigned long long>(floor(static_cast<double>(top_p) * static_cast<double>(total)));
    }
    level_crossing(sh, 255, above, limit);
    __syncthreads();
    const int bin = sh.sel;
    if (!sh.found) {
      keep_all = true;
      __syncthreads();
      break;
    }
    above = sh.sel_above;
    prefix = (prefix << 8) | static_cast<uint32_t>(bin);
    grp_mass = sh.tmass[bin];
    grp_cnt = sh.tcnt[bin];
    __syncthreads();
  }
  if (keep_all) {
    tau_out = 0u;
    cut_out = INT32_MAX;
    K_out = static_cast<double>(total) * kInv40;
    return;
  }
  // A bf16 logit's 32-bit key has 16 low bits that are all zero (value >= 0)
  // or all one (value < 0: the key is the complement of the bits).
  const uint32_t tau = sizeof(E) == 2 ? ((prefix << 16) | ((prefix & 0x8000u) ? 0u : 0xffffu)) : prefix;
  const unsigned long long e_tau = grp_mass / grp_cnt;
  unsigned long long nk = (limit - above) / e_tau + 1;
  int32_t cut = INT32_MAX;
  if (nk < grp_cnt) {
    uint32_t sp = 0;
    unsigned need = static_cast<unsigned>(nk);
#pragma unroll 1
    for (int q = 0; q < 3; ++q, ++pass_no) {
      const int buf = pass_no & 1;
      const int sb = 16 - 8 * q;
      for (int t = threadIdx.x; t < 4 * 256; t += kTpThreads) (&sh.lvl[buf][0][0])[t] = 0u;
      __syncthreads();
      for_slice<E, NV>(row, S.len, rank, [&](float x, int j) {
        if (order_key(x) != tau) return;
        const uint32_t s2 = static_cast<uint32_t>(tie_key(S, j));
        if (q == 0 || (s2 >> (sb + 8)) == sp) atomicAdd(&sh.lvl[buf][0][(s2 >> sb) & 255], 1u);
      });
      reduce_levels(cluster, sh, buf, cl);
      count_crossing(sh, need);
      __syncthreads();
      sp = (sp << 8) | static_cast<uint32_t>(sh.sel);
      need -= static_cast<unsigned>(sh.sel_above);
      __syncthreads();
    }
    cut = static_cast<int32_t>(sp);
  } else {
    nk = grp_cnt;
  }
  tau_out = tau;
  cut_out = cut;
  K_out = static_cast<double>(above + nk * e_tau) * kInv40;
}

template <typename E, int NV>
__global__ void __launch_bounds__(kTpThreads, 2) topp_stats_kernel(StatsLaunch L) {
  constexpr int EPV = Elem<E>::kPerVec;
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  TpShared& sh = *reinterpret_cast<TpShared*>(dyn_smem);
  cg::cluster_group cluster = cg::this_cluster();
  const int cl = L.cl;
  const int rank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x;
  int r = blockIdx.x / cl;
  const RowSet& S = pick_set(L, r);
  const E* row = reinterpret_cast<const E*>(S.base) + static_cast<int64_t>(r) * S.stride;
  const float c = L.c;

  // 1. Row in registers; cluster maximum.
  RowRegs<E, NV> R;
  float lm = load_row_regs<E, NV>(R, row, S.len, rank);
  if (tid == 0) {
    sh.gn = 0;
    sh.cn = 0;
    sh.flags = 0;
  }
  lm = block_max<kTpThreads>(lm, sh.red_f);
  if (tid == 0) sh.cta_max = lm;
  __syncthreads();
  cluster.sync();
  float M = -CUDART_INF_F;
  {
    // Lane q of every warp reads block q's maximum; one warp reduction.
    const int lane = tid & 31;
    float v = lane < cl ? cluster.map_shared_rank(&sh, lane)->cta_max : -CUDART_INF_F;
    M = warp_max(v);
  }
  const float mc = M * c;
  const bool empty = !(M > -CUDART_INF_F);

  uint32_t tau = 0u;
  int32_t cut = INT32_MAX;
  double K = 0.0;
  int pass_no = 0;
  bool generic = false;
  if (!empty) {
    // 2. Pass A: private per-thread bin masses.
    float* ph = sh.phist;
#pragma unroll 4
    for (int b = 0; b < kNB; ++b) ph[b * kTpThreads + tid] = 0.0f;
    auto add_a = [&](float x) {
      const float e = weight(x, c, mc);
      const int b = mass_bin(e);
      ph[b * kTpThreads + tid] += e;
    };
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int i = 0; i < EPV; ++i) add_a(R.val(k, i));
    if (R.xi >= 0) add_a(R.xv);
    __syncthreads();
    {
      // Block totals per bin: 4 threads per bin, each summing 64 columns.
      const int b = tid >> 2, part = tid & 3;
      float s = 0.0f;
#pragma unroll 8
      // Rotated column order: the 32 lanes of a warp hit 32 different banks.
      for (int t = 0; t < 64; ++t) s += ph[b * kTpThreads + part * 64 + ((t + 4 * (b & 7) + part) & 63)];
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (part == 0) sh.cta_bins[b] = s;
    }
    __syncthreads();
    cluster.sync();
    if (tid < 32) {
      // Warp 0: row totals of bins 2*lane and 2*lane+1 (all remote loads
      // issued at once), then a scan from the top bin down.
      double r0 = 0.0, r1 = 0.0;
      {
        float v0[16], v1[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          if (q < cl) {
            const TpShared* p = cluster.map_shared_rank(&sh, q);
            v0[q] = p->cta_bins[2 * tid];
            v1[q] = p->cta_bins[2 * tid + 1];
          } else {
            v0[q] = v1[q] = 0.0f;
          }
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          r0 += static_cast<double>(v0[q]);
          r1 += static_cast<double>(v1[q]);
        }
      }
      const double pair = r0 + r1;
      double incl = pair;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      const double tot = __shfl_sync(0xffffffffu, incl, 31);
      const double lim = static_cast<double>(L.top_p) * tot;
      const double before = incl - pair;
      int hit = -1;
      double a0 = 0.0;
      if (before + r0 > lim) {
        hit = 2 * tid;
        a0 = before;
      } else if (before + pair > lim) {
        hit = 2 * tid + 1;
        a0 = before + r0;
      }
      const unsigned hb = __ballot_sync(0xffffffffu, hit >= 0);
      const int src = hb ? __ffs(hb) - 1 : 0;
      const int bs = hb ? __shfl_sync(0xffffffffu, hit, src) : -1;
      const double a = __shfl_sync(0xffffffffu, a0, src);
      if (tid == 0) {
        sh.total = tot;
        sh.limit = lim;
        sh.bstar = bs;
        sh.above0 = a;
      }
    }
    __syncthreads();
    const double total = sh.total;
    const double limit = sh.limit;
    const int bstar = sh.bstar;
    const double above0 = sh.above0;
    if (bstar < 0) {
      K = total;  // nothing exceeds top_p: every id is kept
    } else if (bstar == kNB - 1) {
      generic = true;
    } else {
      // 3. Pass B: candidates of bin b*, level-1 histogram on e bits 21..14.
      // Each warp owns a region of the candidate list and a private copy of
      // the level-1 histogram (in the now unused pass-A histogram space), so
      // no two warps contend for one address.  Level masses are fixed point
      // relative to bin b*: e * 2^(30 + floor(b*/2)) < 2^31.
      constexpr int kWarps = kTpThreads / 32;
      constexpr int kCapW = kCap / kWarps;
      const int warp = tid >> 5, lane = tid & 31;
      const unsigned lane_lt = (1u << lane) - 1u;
      const float lscale = ldexpf(1.0f, 30 + bstar / 2);
      unsigned* wl = reinterpret_cast<unsigned*>(sh.phist) + warp * 3 * 256;  // [count, lo, hi][256]
      for (int t = lane; t < 3 * 256; t += 32) wl[t] = 0u;
      for (int t = tid; t < 256; t += kTpThreads) sh.lvl[0][3][t] = 0u;
      __syncwarp();
      int wbase = 0;
      auto add_b = [&](float x, int j) {
        const float e = ex2v(fmaf(x, c, -mc));
        const bool cand = j >= 0 && mass_bin(e) == bstar;
        const unsigned bal = __ballot_sync(0xffffffffu, cand);
        if (cand) {
          const uint32_t eb = __float_as_uint(e);
          const int sub = (eb >> 14) & 255;
          const unsigned v = __float2uint_rn(e * lscale);
          atomicAdd(&wl[sub], 1u);
          atomicAdd(&wl[256 + sub], v & 0xffffu);
          atomicAdd(&wl[512 + sub], v >> 16);
          const int slot = wbase + __popc(bal & lane_lt);
          if (slot < kCapW) {
            sh.cbits[warp * kCapW + slot] = __float_as_uint(x);
            sh.csec[warp * kCapW + slot] = tie_key(S, j);
          }
        }
        wbase += __popc(bal);
      };
#pragma unroll
      for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int i = 0; i < EPV; ++i) {
          const int j = R.idx(k, i);
          add_b(R.val(k, i), j < S.len ? j : -1);
        }
      add_b(R.xv, R.xi);
      if (lane == 0) sh.wcnt[warp] = wbase;
      __syncthreads();
      // Merge the warp histograms; pack the warp regions into one list.
      for (int t = tid; t < 256; t += kTpThreads) {
        unsigned cnt = 0, lo = 0, hi = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const unsigned* h = reinterpret_cast<const unsigned*>(sh.phist) + w * 3 * 256;
          cnt += h[t];
          lo += h[256 + t];
          hi += h[512 + t];
        }
        sh.lvl[0][0][t] = cnt;
        sh.lvl[0][1][t] = lo;
        sh.lvl[0][2][t] = hi;
      }
      int over = 0, total_c = 0, my_off = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int n = sh.wcnt[w];
        over |= n > kCapW;
        if (w < warp) my_off += n;
        total_c += n;
      }
      // Compaction into the front of the list: warps move their entries in
      // order (a warp's destination never overlaps a later warp's source).
      for (int w = 1; w < kWarps; ++w) {
        __syncthreads();
        if (warp == w && !over) {
          const int n = sh.wcnt[w];
          for (int e2 = lane; e2 < n; e2 += 32) {
            sh.cbits[my_off + e2] = sh.cbits[w * kCapW + e2];
            sh.csec[my_off + e2] = sh.csec[w * kCapW + e2];
          }
        }
      }
      __syncthreads();
      if (tid == 0) {
        sh.cn = over ? kCap + 1 : total_c;
        if (over) sh.flags |= 1;
      }
      __syncthreads();
      cluster.sync();
      int any_over = 0;
      {
        const int f = lane < cl ? cluster.map_shared_rank(&sh, lane)->flags : 0;
        any_over = __any_sync(0xffffffffu, f != 0) ? 1 : 0;
      }
      if (any_over) {
        generic = true;
      } else {
        // Levels: e bits 21..14, 13..6, 5..0.
        const unsigned long long lim_fixed =
            limit > above0 ? static_cast<unsigned long long>((limit - above0) * static_cast<double>(lscale)) : 0ull;
        unsigned long long above_fixed = 0;
        uint32_t pref = 255u - static_cast<uint32_t>(bstar);  // e bits >> 22
        // Level l histograms e bits [shift(l), shift(l) + width(l)).
        auto shift_of = [](int l) { return l == 0 ? 14 : (l == 1 ? 6 : 0); };
        auto width_of = [](int l) { return l == 2 ? 6 : 8; };
        int lvl = 0;
        unsigned grp = 0;
        pass_no = 0;
        bool done_levels = false;
        while (!done_levels) {
          const int buf = pass_no & 1;
          reduce_levels(cluster, sh, buf, cl);
          level_crossing(sh, (1 << width_of(lvl)) - 1, above_fixed, lim_fixed);
          __syncthreads();
          const int sel = sh.sel;
          above_fixed = sh.sel_above;
          grp = sh.sel_cnt;
          pref = (pref << width_of(lvl)) | static_cast<uint32_t>(sel);
          __syncthreads();
          if (grp <= static_cast<unsigned>(kFinal) || lvl == 2) {
            done_levels = true;
          } else {
            ++lvl;
            ++pass_no;
            const int nb = pass_no & 1;
            for (int t = tid; t < 4 * 256; t += kTpThreads) (&sh.lvl[nb][0][0])[t] = 0u;
            __syncthreads();
            const int cn = sh.cn;
            for (int s = tid; s < cn; s += kTpThreads) {
              const float x = __uint_as_float(sh.cbits[s]);
              const float e = ex2v(fmaf(x, c, -mc));
              const uint32_t eb = __float_as_uint(e);
              if ((eb >> (shift_of(lvl) + width_of(lvl))) != pref) continue;
              const int sub = (eb >> shift_of(lvl)) & ((1 << width_of(lvl)) - 1);
              const unsigned v = __float2uint_rn(e * lscale);
              atomicAdd(&sh.lvl[nb][0][sub], 1u);
              atomicAdd(&sh.lvl[nb][1][sub], v & 0xffffu);
              atomicAdd(&sh.lvl[nb][2][sub], v >> 16);
            }
          }
        }
        const int fshift = shift_of(lvl);
        const double above = above0 + static_cast<double>(above_fixed) / static_cast<double>(lscale);
        if (grp <= static_cast<unsigned>(kFinal)) {
          // 4. Gather the final group into the first block and sort it.
          TpShared* r0 = cluster.map_shared_rank(&sh, 0);
          const int cn = sh.cn;
          for (int s = tid; s < cn; s += kTpThreads) {
            const float x = __uint_as_float(sh.cbits[s]);
            const uint32_t eb = __float_as_uint(weight(x, c, mc));
            if ((eb >> fshift) != pref) continue;
            const int slot = atomicAdd(&r0->gn, 1);
            if (slot < kFinal) {
              r0->gbits[slot] = sh.cbits[s];
              r0->gsec[slot] = sh.csec[s];
            }
          }
          __syncthreads();
          cluster.sync();
          if (rank == 0 && tid < 32) {
            const int n = min(sh.gn, kFinal);
            unsigned long long a = 0, b = 0;
            if (tid < n)
              a = (static_cast<unsigned long long>(order_key(__uint_as_float(sh.gbits[tid]))) << 32) |
                  (0xffffffffu - static_cast<uint32_t>(sh.gsec[tid]));
            if (tid + 32 < n)
              b = (static_cast<unsigned long long>(order_key(__uint_as_float(sh.gbits[tid + 32]))) << 32) |
                  (0xffffffffu - static_cast<uint32_t>(sh.gsec[tid + 32]));
            int ra = 0, rb = 0;
#pragma unroll 4
            for (int j = 0; j < 32; ++j) {
              const unsigned long long xa = __shfl_sync(0xffffffffu, a, j);
              const unsigned long long xb = __shfl_sync(0xffffffffu, b, j);
              ra += (xa > a) + (xb > a);
              rb += (xa > b) + (xb > b);
            }
            // Sorted order: composite keys are distinct for distinct ids.
            __syncwarp();
            uint32_t gb0 = tid < n ? sh.gbits[tid] : 0u, gb1 = tid + 32 < n ? sh.gbits[tid + 32] : 0u;
            int32_t gs0 = tid < n ? sh.gsec[tid] : 0, gs1 = tid + 32 < n ? sh.gsec[tid + 32] : 0;
            __syncwarp();
            if (tid < n) {
              sh.gbits[ra] = gb0;
              sh.gsec[ra] = gs0;
            }
            if (tid + 32 < n) {
              sh.gbits[rb] = gb1;
              sh.gsec[rb] = gs1;
            }
            __syncwarp();
            if (tid == 0) {
              double cum = above;
              int pick = n - 1;
#pragma unroll 1
              for (int j = 0; j < n; ++j) {
                const double e = static_cast<double>(weight(__uint_as_float(sh.gbits[j]), c, mc));
                if (cum + e > limit) {
                  pick = j;
                  break;
                }
                cum += e;
              }
              double kept_mass = above;
#pragma unroll 1
              for (int j = 0; j <= pick; ++j)
                kept_mass += static_cast<double>(weight(__uint_as_float(sh.gbits[j]), c, mc));
              tau = order_key(__uint_as_float(sh.gbits[pick]));
              cut = sh.gsec[pick];
              K = kept_mass;
            }
          }
        } else {
          // More than kFinal elements share one value of e.  Equal logits: cut
          // the tie group by its tie keys; otherwise the generic path.
          uint32_t kmin = 0xffffffffu, kmax = 0u;
          const int cn = sh.cn;
          for (int s = tid; s < cn; s += kTpThreads) {
            const float x = __uint_as_float(sh.cbits[s]);
            const uint32_t eb = __float_as_uint(weight(x, c, mc));
            if ((eb >> fshift) != pref) continue;
            const uint32_t key = order_key(x);
            kmin = min(kmin, key);
            kmax = max(kmax, key);
          }
          kmin = block_min_u32<kTpThreads>(kmin, sh.red_u);
          kmax = static_cast<uint32_t>(block_max_u64<kTpThreads>(kmax, sh.red_u));
          if (tid == 0) {
            sh.kmin = kmin;
            sh.kmax = kmax;
          }
          __syncthreads();
          cluster.sync();
          {
            const int lane = tid & 31;
            uint32_t a = 0xffffffffu, z = 0u;
            if (lane < cl) {
              const TpShared* p = cluster.map_shared_rank(&sh, lane);
              a = p->kmin;
              z = p->kmax;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
              z = max(z, __shfl_xor_sync(0xffffffffu, z, o));
            }
            kmin = min(kmin, a);
            kmax = max(kmax, z);
          }
          if (kmin != kmax) {
            generic = true;
          } else {
            const float xv = __uint_as_float(kmin & 0x80000000u ? (kmin & 0x7fffffffu) : ~kmin);
            const double e_g = static_cast<double>(weight(xv, c, mc));
            double nkd = floor((limit - above) / e_g) + 1.0;
            if (!(nkd >= 1.0)) nkd = 1.0;
            unsigned nk = nkd >= static_cast<double>(grp) ? grp : static_cast<unsigned>(nkd);
            tau = kmin;
            K = above + static_cast<double>(nk) * e_g;
            if (nk < grp) {
              uint32_t sp = 0;
              unsigned need = nk;
              for (int q = 0; q < 3; ++q) {
                ++pass_no;
                const int b2 = pass_no & 1;
                const int sb = 16 - 8 * q;
                for (int t = tid; t < 4 * 256; t += kTpThreads) (&sh.lvl[b2][0][0])[t] = 0u;
                __syncthreads();
                for (int s = tid; s < cn; s += kTpThreads) {
                  if (order_key(__uint_as_float(sh.cbits[s])) != tau) continue;
                  const uint32_t s2 = static_cast<uint32_t>(sh.csec[s]);
                  if (q == 0 || (s2 >> (sb + 8)) == sp) atomicAdd(&sh.lvl[b2][0][(s2 >> sb) & 255], 1u);
                }
                reduce_levels(cluster, sh, b2, cl);
                count_crossing(sh, need);
                __syncthreads();
                sp = (sp << 8) | static_cast<uint32_t>(sh.sel);
                need -= static_cast<unsigned>(sh.sel_above);
                __syncthreads();
              }
              cut = static_cast<int32_t>(sp);
            }
          }
        }
      }
    }
    if (generic) {
      ++pass_no;
      generic_select<E, NV>(cluster, sh, row, S, rank, cl, c, mc, L.top_p, pass_no, tau, cut, K);
    }
  }
  if (rank == 0 && tid == 0) {
    RowStats st;
    st.m = M;
    st.mc = mc;
    st.tau = tau;
    st.cut = cut;
    st.K = K;
    st.status = empty ? SV_ROW_EMPTY : 0u;
    st.e_query = 0.0f;
    const Query q = row_query(S, r);
    if (q.bad) st.status |= SV_ROW_BAD_DRAFT_ID;
    if (q.elem >= 0 && !empty) {
      const float x = Elem<E>::load(row + q.elem);
      if (kept(order_key(x), q.sec, tau, cut)) st.e_query = weight(x, c, mc);
    }
    S.out[r] = st;
  }
  // No block may leave while a peer can still read its shared memory.
  cluster.sync();
}

template <typename E, int NV>
static sv_status launch_nv(const StatsLaunch& L, int rows, cudaStream_t stream) {
  auto kern = topp_stats_kernel<E, NV>;
  static FuncAttrCache cache;
  const size_t smem = sizeof(TpShared);
  if (!cache.ensure(reinterpret_cast<const void*>(kern), smem, L.cl > 8)) return SV_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(rows) * L.cl);
  cfg.blockDim = dim3(kTpThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(L.cl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, L) != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

// Vectors per thread and cluster size for rows of at most max_len elements:
// the smallest cluster whose blocks need at most 12 vectors per thread (the
// row then stays in registers with two blocks per SM).
template <typename E>
static sv_status launch_topp_typed(StatsLaunch L, int rows, int max_len, cudaStream_t stream) {
  constexpr int EPV = Elem<E>::kPerVec;
  // An unaligned row has a scalar head, so its body never exceeds ceil(len/EPV) vectors.
  const int nvec = (max_len + EPV - 1) / EPV;
  int cl = 1;
  while (cl < 16 && (nvec + cl * kTpThreads - 1) / (cl * kTpThreads) > 12) cl *= 2;
  const int per = (nvec + cl * kTpThreads - 1) / (cl * kTpThreads);
  if (per > 12) return SV_ERR_UNSUPPORTED;
  L.cl = cl;
  if (per <= 4) return launch_nv<E, 4>(L, rows, stream);
  if (per <= 8) return launch_nv<E, 8>(L, rows, stream);
  return launch_nv<E, 12>(L, rows, stream);
}

sv_status launch_topp_stats(const StatsLaunch& L, int rows, int max_len, sv_dtype dtype, cudaStream_t stream) {
  if (rows == 0) return SV_OK;
  return dtype == SV_BF16 ? launch_topp_typed<uint16_t>(L, rows, max_len, stream)
                          : launch_topp_typed<float>(L, rows, max_len, stream);
}

}  // namespace sv
