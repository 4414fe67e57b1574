// Row statistics with the top-p (nucleus) threshold, for temperature > 0 and
// top_p < 1.
//
// Source: "LLM inference acceleration in practice: draft models and
// speculative sampling explained" (mlqm.cn), §4.2 _apply_top_p: rank the
// logits in descending order, keep rank r iff r == 0 or the softmax mass of
// the ranks before it is at most top_p; equal logits are ranked by lower
// index (EAGLE3 draft rows: by target id).
//
// Work split, without clusters and without any block waiting for another:
//  * slice blocks: every block reads one slice of 8192 logits of a row into
//    registers, takes the slice maximum m_s, and adds e_s = 2^(l*c - m_s*c)
//    (c = log2(e)/T) to a per-thread private histogram keyed by the ABSOLUTE
//    half-octave g = floor(2*l*c) of the logit ([bin][thread] layout, no
//    atomics).  It publishes (m_s, bins, mass below the bins) and bumps the
//    row's counter;
//  * the row's last slice block merges the summaries (absolute bins line up
//    across slices after scaling by 2^((m_s - m)*c)), finds the half-octave
//    g* where the cumulative mass from the top first exceeds top_p * S, then
//    rescans the row (just read by its sibling blocks, so served by L2) for
//    the logits of g*, refines them on finer sub-bins of 2*l*c in shared
//    memory, and resolves the last <= 64 exactly: sorted by (logit
//    descending, tie key ascending), walked in double precision.
// Rare rows (the cut below the 64 half-octaves under the maximum, more than
// 16384 candidates, or a large group of different logits that 2*l*c cannot
// separate) take an exact radix select over the order keys of the row.
#include "sv_rows.cuh"

namespace sv {

constexpr int kSThreads = 256;
constexpr int kSEPT = 32;                       // logits per thread per slice
constexpr int kSlice = kSThreads * kSEPT;       // logits per slice
constexpr int kGB = 64;                         // half-octave bins below the maximum
constexpr int kSummary = 4 + kGB;               // floats per slice summary
constexpr int kListCap = 16384;                 // candidate indices in shared memory
constexpr int kFinal = 64;
constexpr int kWarps = kSThreads / 32;
constexpr double kScale40 = 1099511627776.0;    // generic path: masses in units of 2^-40
constexpr double kInv40 = 1.0 / 1099511627776.0;

struct ToppShared {
  union {
    float phist[kGB * kSThreads];               // slice phase: private bin masses
    int list[kListCap];                         // merge phase: candidate indices
  };
  unsigned wl[kWarps][3][256];                  // per-warp level histograms (count, lo, hi)
  unsigned long long tmass[256];
  unsigned tcnt[256];
  float mbins[kWarps][kGB];
  float mfar[kWarps];
  float red_f[32];
  unsigned long long red_u[32];
  int gidx[kFinal];
  int wcnt[kWarps];
  int last;
  int cn;
  int sel;
  int found;
  unsigned long long sel_above;
  unsigned sel_cnt;
  int gstar;
  int pick_sec;
  unsigned pick_key;
  double above0, limit, total, kept_mass;
};

// exp2 that the compiler may not merge with an identical earlier one.
__device__ __forceinline__ float ex2v(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Absolute half-octave of a logit: floor(2 * l * c).  The same expression
// everywhere, so membership is decided identically in every pass.
__device__ __forceinline__ int half_octave(float l, float c) { return __float2int_rd(2.0f * (l * c)); }

template <typename E>
__device__ __forceinline__ float widen(const uint4& v, int i) {
  if constexpr (sizeof(E) == 4) {
    return Elem<E>::at(v, i);
  } else {
    // Volatile so that every pass widens again instead of keeping 2x data live.
    const uint32_t w = (i >> 1) == 0 ? v.x : (i >> 1) == 1 ? v.y : (i >> 1) == 2 ? v.z : v.w;
    uint32_t r;
    if (i & 1) asm volatile("and.b32 %0, %1, 0xffff0000;" : "=r"(r) : "r"(w));
    else asm volatile("shl.b32 %0, %1, 16;" : "=r"(r) : "r"(w));
    return __uint_as_float(r);
  }
}

// Visit every logit of a row (body vectors strided over the block, then the
// scalar head and tail): f(value, index), index -1 for padding.
template <typename E, typename F>
__device__ __forceinline__ void for_row(const E* row, int len, F&& f) {
  constexpr int EPV = Elem<E>::kPerVec;
  const RowSplit rs = split_row(row, len);
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  constexpr int U = 4;
  // Block-uniform trip count: f may use full-warp votes.
  for (int base = 0; base < rs.nvec; base += kSThreads * U) {
    const int v0 = base + static_cast<int>(threadIdx.x);
    uint4 w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * kSThreads;
      w[u] = v < rs.nvec ? __ldcg(vp + v) : Elem<E>::neg_inf_vec();
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + u * kSThreads;
#pragma unroll
      for (int i = 0; i < EPV; ++i) f(Elem<E>::at(w[u], i), v < rs.nvec ? rs.head + v * EPV + i : -1);
    }
  }
  const int ntail = len - rs.tail0;
  // Every thread runs the same number of iterations (f may use warp votes).
  for (int t0 = 0; t0 < rs.head + ntail; t0 += kSThreads) {
    const int t = t0 + static_cast<int>(threadIdx.x);
    const int j = t < rs.head ? t : (t < rs.head + ntail ? rs.tail0 + (t - rs.head) : -1);
    f(j >= 0 ? Elem<E>::load(row + j) : -CUDART_INF_F, j);
  }
}

// Warp 0: first bin from `top` down to 0 where above + mass > limit; if none,
// the lowest non-empty bin.  Bins come from sh.tmass / sh.tcnt.
__device__ __forceinline__ void crossing_desc(ToppShared& sh, int top, unsigned long long above,
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
  int b;
  unsigned long long a;
  if (hb) {
    const int src = __ffs(hb) - 1;
    b = __shfl_sync(0xffffffffu, hit, src);
    a = __shfl_sync(0xffffffffu, hit_above, src);
  } else {
    const int src = lb ? 31 - __clz(lb) : 0;
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
__device__ __forceinline__ void crossing_count(ToppShared& sh, unsigned need) {
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

__device__ __forceinline__ void clear_wl(ToppShared& sh) {
  unsigned* w = &sh.wl[0][0][0];
  for (int t = threadIdx.x; t < kWarps * 3 * 256; t += kSThreads) w[t] = 0u;
}

// Merge the per-warp level histograms into sh.tmass / sh.tcnt.
__device__ __forceinline__ void merge_wl(ToppShared& sh) {
  for (int t = threadIdx.x; t < 256; t += kSThreads) {
    unsigned long long lo = 0, hi = 0;
    unsigned cnt = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      cnt += sh.wl[w][0][t];
      lo += sh.wl[w][1][t];
      hi += sh.wl[w][2][t];
    }
    sh.tcnt[t] = cnt;
    sh.tmass[t] = lo + (hi << 16);
  }
}

template <typename E>
__device__ __forceinline__ float load_at(const E* row, int j) {
  if constexpr (sizeof(E) == 4) return __ldcg(reinterpret_cast<const float*>(row) + j);
  else return __uint_as_float(static_cast<uint32_t>(__ldcg(reinterpret_cast<const unsigned short*>(row) + j)) << 16);
}

// Exact path for rare rows: radix select over the 32-bit order keys of the
// whole row with (count, 40-bit fixed-point mass) histograms, then the tie
// cut over tie keys.  One block, reading the row from global memory.
template <typename E>
__device__ __noinline__ void generic_select(ToppShared& sh, const E* row, const RowSet& S, float c, float mc,
                                            float top_p, uint32_t& tau_out, int32_t& cut_out, double& K_out) {
  constexpr int kPasses = sizeof(E) == 2 ? 2 : 4;
  unsigned* h = &sh.wl[0][0][0];  // [count, m0, m1, m2][256]
  uint32_t prefix = 0;
  unsigned long long above = 0, limit = 0, total = 0, grp_mass = 0;
  unsigned grp_cnt = 0;
  bool keep_all = false;
#pragma unroll 1
  for (int p = 0; p < kPasses; ++p) {
    const int sb = 24 - 8 * p;
    for (int t = threadIdx.x; t < 4 * 256; t += kSThreads) h[t] = 0u;
    __syncthreads();
    for_row<E>(row, S.len, [&](float x, int j) {
      if (j < 0) return;
      const uint32_t key = order_key(x);
      if (p == 0 || (key >> (sb + 8)) == prefix) {
        const int bin = (key >> sb) & 255;
        const unsigned long long v =
            __double2ull_rn(static_cast<double>(ex2v(fmaf(x, c, -mc))) * kScale40);
        atomicAdd(&h[bin], 1u);
        if (v) {
          atomicAdd(&h[256 + bin], static_cast<unsigned>(v & 0xffffu));
          atomicAdd(&h[512 + bin], static_cast<unsigned>((v >> 16) & 0xffffu));
          atomicAdd(&h[768 + bin], static_cast<unsigned>(v >> 32));
        }
      }
    });
    __syncthreads();
    for (int t = threadIdx.x; t < 256; t += kSThreads) {
      sh.tcnt[t] = h[t];
      sh.tmass[t] = static_cast<unsigned long long>(h[256 + t]) +
                    (static_cast<unsigned long long>(h[512 + t]) << 16) +
                    (static_cast<unsigned long long>(h[768 + t]) << 32);
    }
    __syncthreads();
    if (p == 0) {
      unsigned long long part = 0;
      for (int t = threadIdx.x; t < 256; t += kSThreads) part += sh.tmass[t];
      total = block_sum_u64<kSThreads>(part, sh.red_u);
      limit = static_cast<unsigned long long>(floor(static_cast<double>(top_p) * static_cast<double>(total)));
    }
    crossing_desc(sh, 255, above, limit);
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
    for (int q = 0; q < 3; ++q) {
      const int sb = 16 - 8 * q;
      for (int t = threadIdx.x; t < 256; t += kSThreads) h[t] = 0u;
      __syncthreads();
      for_row<E>(row, S.len, [&](float x, int j) {
        if (j < 0 || order_key(x) != tau) return;
        const uint32_t s2 = static_cast<uint32_t>(tie_key(S, j));
        if (q == 0 || (s2 >> (sb + 8)) == sp) atomicAdd(&h[(s2 >> sb) & 255], 1u);
      });
      __syncthreads();
      for (int t = threadIdx.x; t < 256; t += kSThreads) sh.tcnt[t] = h[t];
      __syncthreads();
      crossing_count(sh, need);
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

// The row's cut from the merged half-octave bins (last slice block only).
// Returns false when the row needs the generic path.
template <typename E>
__device__ bool resolve_row(ToppShared& sh, const E* row, const RowSet& S, float c, float mc, int gstar,
                            double above0, double limit, uint32_t& tau, int32_t& cut, double& K) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lane_lt = (1u << lane) - 1u;
  // Masses of the cut half-octave: e < 2^((g*+1)/2 - mc) <= 2^k, held as
  // e * 2^(30 - k) < 2^30 in fixed point.
  const int k = static_cast<int>(ceilf(0.5f * static_cast<float>(gstar + 1) - mc)) + 1;
  const float lscale = ldexpf(1.0f, 30 - k);
  const float g_lo = static_cast<float>(gstar);
  constexpr int kRegion = kListCap / kWarps;
  // Rescan: candidates of g*, level-1 histogram on floor(256 * (2lc - g*)).
  clear_wl(sh);
  __syncthreads();
  int wbase = 0;
  for_row<E>(row, S.len, [&](float x, int j) {
    const bool cand = j >= 0 && half_octave(x, c) == gstar;
    const unsigned bal = __ballot_sync(0xffffffffu, cand);
    if (cand) {
      const float u = 2.0f * (x * c) - g_lo;
      const int s1 = min(255, max(0, static_cast<int>(u * 256.0f)));
      const unsigned v = __float2uint_rn(ex2v(fmaf(x, c, -mc)) * lscale);
      atomicAdd(&sh.wl[warp][0][s1], 1u);
      atomicAdd(&sh.wl[warp][1][s1], v & 0xffffu);
      atomicAdd(&sh.wl[warp][2][s1], v >> 16);
      const int slot = wbase + __popc(bal & lane_lt);
      if (slot < kRegion) sh.list[warp * kRegion + slot] = j;
    }
    wbase += __popc(bal);
  });
  if (lane == 0) sh.wcnt[warp] = wbase;
  __syncthreads();
  merge_wl(sh);
  int over = 0, cn = 0, my_off = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int n = sh.wcnt[w];
    over |= n > kRegion;
    if (w < warp) my_off += n;
    cn += n;
  }
  if (over) return false;  // uniform: every thread read the same counts
  // Pack the warp regions into the front of the list, in warp order (a
  // warp's destination never overlaps a later warp's region).
  for (int w = 1; w < kWarps; ++w) {
    __syncthreads();
    if (warp == w) {
      const int n = sh.wcnt[w];
      for (int e2 = lane; e2 < n; e2 += 32) sh.list[my_off + e2] = sh.list[w * kRegion + e2];
    }
  }
  __syncthreads();
  const unsigned long long lim_fixed =
      limit > above0 ? static_cast<unsigned long long>((limit - above0) * static_cast<double>(lscale)) : 0ull;
  unsigned long long above_fixed = 0;
  // Levels: sub-bin floor(256^(L+1) * (2lc - g*)) with the earlier digits fixed.
  int pref = 0;
  for (int lvl = 0;; ++lvl) {
    crossing_desc(sh, 255, above_fixed, lim_fixed);
    __syncthreads();
    const int sel = sh.sel;
    above_fixed = sh.sel_above;
    const unsigned grp = sh.sel_cnt;
    pref = pref * 256 + sel;
    const float scale_l = lvl == 0 ? 256.0f : (lvl == 1 ? 65536.0f : 16777216.0f);
    __syncthreads();
    {
      // Keep only the chosen sub-bin, order preserved: chunks of one entry
      // per thread, block-wide scan of the keep flags, in-place writes (a
      // chunk is read completely before any of it is written).
      int kept_n = 0;
      for (int b0 = 0; b0 < cn; b0 += kSThreads) {
        const int s = b0 + tid;
        bool keep = false;
        int jv = 0;
        if (s < cn) {
          jv = sh.list[s];
          const float u = 2.0f * (load_at<E>(row, jv) * c) - g_lo;
          keep = static_cast<int>(u * scale_l) == pref;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (lane == 0) sh.wcnt[warp] = __popc(bal);
        __syncthreads();
        int off = kept_n, chunk = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const int n = sh.wcnt[w];
          if (w < warp) off += n;
          chunk += n;
        }
        if (keep) sh.list[off + __popc(bal & lane_lt)] = jv;
        kept_n += chunk;
        __syncthreads();
      }
      if (tid == 0) sh.cn = kept_n;
    }
    __syncthreads();
    cn = sh.cn;
    if (grp <= static_cast<unsigned>(kFinal) || lvl == 2) break;
    const float scale_n = lvl == 0 ? 65536.0f : 16777216.0f;
    clear_wl(sh);
    __syncthreads();
    for (int s = tid; s < cn; s += kSThreads) {
      const int jv = sh.list[s];
      const float x = load_at<E>(row, jv);
      const float u = 2.0f * (x * c) - g_lo;
      const int sb = min(255, max(0, static_cast<int>(u * scale_n) - pref * 256));
      const unsigned v = __float2uint_rn(ex2v(fmaf(x, c, -mc)) * lscale);
      atomicAdd(&sh.wl[warp][0][sb], 1u);
      atomicAdd(&sh.wl[warp][1][sb], v & 0xffffu);
      atomicAdd(&sh.wl[warp][2][sb], v >> 16);
    }
    __syncthreads();
    merge_wl(sh);
    __syncthreads();
  }
  const double above = above0 + static_cast<double>(above_fixed) / static_cast<double>(lscale);
  if (cn <= kFinal) {
    // Sort the final group by (logit descending, tie key ascending), walk it.
    if (warp == 0) {
      unsigned long long a = 0, b = 0;
      int ja = -1, jb = -1;
      if (lane < cn) {
        ja = sh.list[lane];
        a = (static_cast<unsigned long long>(order_key(load_at<E>(row, ja))) << 32) |
            (0xffffffffu - static_cast<uint32_t>(tie_key(S, ja)));
      }
      if (lane + 32 < cn) {
        jb = sh.list[lane + 32];
        b = (static_cast<unsigned long long>(order_key(load_at<E>(row, jb))) << 32) |
            (0xffffffffu - static_cast<uint32_t>(tie_key(S, jb)));
      }
      int ra = 0, rb = 0;
#pragma unroll 4
      for (int j2 = 0; j2 < 32; ++j2) {
        const unsigned long long xa2 = __shfl_sync(0xffffffffu, a, j2);
        const unsigned long long xb2 = __shfl_sync(0xffffffffu, b, j2);
        ra += (xa2 > a) + (xb2 > a);
        rb += (xa2 > b) + (xb2 > b);
      }
      if (lane < cn) sh.gidx[ra] = ja;
      if (lane + 32 < cn) sh.gidx[rb] = jb;
      __syncwarp();
      if (lane == 0) {
        double cum = above;
        int pick = cn - 1;
        for (int j2 = 0; j2 < cn; ++j2) {
          const double e = static_cast<double>(weight(load_at<E>(row, sh.gidx[j2]), c, mc));
          if (cum + e > limit) {
            pick = j2;
            break;
          }
          cum += e;
        }
        double kept_mass = above;
        for (int j2 = 0; j2 <= pick; ++j2)
          kept_mass += static_cast<double>(weight(load_at<E>(row, sh.gidx[j2]), c, mc));
        const int jp = sh.gidx[pick];
        sh.pick_key = order_key(load_at<E>(row, jp));
        sh.pick_sec = tie_key(S, jp);
        sh.kept_mass = kept_mass;
      }
    }
    __syncthreads();
    tau = sh.pick_key;
    cut = sh.pick_sec;
    K = sh.kept_mass;
    return true;
  }
  // A group that 2*l*c cannot split: equal logits are cut by tie key;
  // different logits go to the exact generic path.
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int s = tid; s < cn; s += kSThreads) {
    const uint32_t key = order_key(load_at<E>(row, sh.list[s]));
    kmin = min(kmin, key);
    kmax = max(kmax, key);
  }
  kmax = static_cast<uint32_t>(block_max_u64<kSThreads>(kmax, sh.red_u));
  kmin = static_cast<uint32_t>(~block_max_u64<kSThreads>(~static_cast<unsigned long long>(kmin) & 0xffffffffull,
                                                          sh.red_u) & 0xffffffffull);
  if (kmin != kmax) return false;
  const float xv = __uint_as_float(kmin & 0x80000000u ? (kmin & 0x7fffffffu) : ~kmin);
  const double e_g = static_cast<double>(weight(xv, c, mc));
  double nkd = floor((limit - above) / e_g) + 1.0;
  if (!(nkd >= 1.0)) nkd = 1.0;
  const unsigned nk = nkd >= static_cast<double>(cn) ? static_cast<unsigned>(cn) : static_cast<unsigned>(nkd);
  tau = kmin;
  K = above + static_cast<double>(nk) * e_g;
  cut = INT32_MAX;
  if (nk < static_cast<unsigned>(cn)) {
    unsigned* h = &sh.wl[0][0][0];
    uint32_t sp = 0;
    unsigned need = nk;
#pragma unroll 1
    for (int q = 0; q < 3; ++q) {
      const int sb = 16 - 8 * q;
      for (int t = tid; t < 256; t += kSThreads) h[t] = 0u;
      __syncthreads();
      for (int s = tid; s < cn; s += kSThreads) {
        const uint32_t s2 = static_cast<uint32_t>(tie_key(S, sh.list[s]));
        if (q == 0 || (s2 >> (sb + 8)) == sp) atomicAdd(&h[(s2 >> sb) & 255], 1u);
      }
      __syncthreads();
      for (int t = tid; t < 256; t += kSThreads) sh.tcnt[t] = h[t];
      __syncthreads();
      crossing_count(sh, need);
      __syncthreads();
      sp = (sp << 8) | static_cast<uint32_t>(sh.sel);
      need -= static_cast<unsigned>(sh.sel_above);
      __syncthreads();
    }
    cut = static_cast<int32_t>(sp);
  }
  return true;
}

template <typename E>
__global__ void __launch_bounds__(kSThreads, 2) topp_slice_kernel(StatsLaunch L) {
  constexpr int EPV = Elem<E>::kPerVec;
  constexpr int VPT = kSEPT / EPV;          // 16-byte vectors per thread
  constexpr int VPS = VPT * kSThreads;      // vectors per slice
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  ToppShared& sh = *reinterpret_cast<ToppShared*>(dyn_smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Block -> (row set, row, slice); the slices of a row are consecutive.
  int blk = blockIdx.x;
  int set = 0;
  if (L.nsets > 1 && blk >= L.set[0].rows * L.nslices[0]) {
    blk -= L.set[0].rows * L.nslices[0];
    set = 1;
  }
  const RowSet& S = L.set[set];
  const int ns = L.nslices[set];
  const int r = blk / ns, s = blk - r * ns;
  const int grow = (set ? L.set[0].rows : 0) + r;
  const int sbase = (set ? L.set[0].rows * L.nslices[0] : 0) + r * ns;
  const E* row = reinterpret_cast<const E*>(S.base) + static_cast<int64_t>(r) * S.stride;
  const float c = L.c;

  // 1. The slice in registers; slice maximum.
  const RowSplit rs = split_row(row, S.len);
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  // Normal L2 policy (not the streaming evict-first one): the row's last
  // block rescans this slice from L2.
  uint4 raw[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = s * VPS + k * kSThreads + tid;
    raw[k] = v < rs.nvec ? __ldcg(vp + v) : Elem<E>::neg_inf_vec();
  }
  float xv = -CUDART_INF_F;
  if (s == 0) {
    const int ntail = S.len - rs.tail0;
    int xi = -1;
    if (tid < rs.head) xi = tid;
    else if (tid < rs.head + ntail) xi = rs.tail0 + (tid - rs.head);
    if (xi >= 0) xv = Elem<E>::load(row + xi);
  }
  float lm = xv;
#pragma unroll
  for (int k = 0; k < VPT; ++k)
#pragma unroll
    for (int i = 0; i < EPV; ++i) lm = fmaxf(lm, Elem<E>::at(raw[k], i));
  const float ms = block_max<kSThreads>(lm, sh.red_f);

  // 2. e relative to the slice maximum, binned by absolute half-octave.
  float* ph = sh.phist;
#pragma unroll 8
  for (int b = 0; b < kGB; ++b) ph[b * kSThreads + tid] = 0.0f;
  const bool live = ms > -CUDART_INF_F;
  const int Gs = live ? half_octave(ms, c) : 0;
  const float mcs = ms * c;
  float far = 0.0f;
  auto add = [&](float x) {
    const float e = ex2(fmaf(x, c, -mcs));
    const int loc = Gs - half_octave(x, c);
    if (loc >= 0 && loc < kGB) ph[loc * kSThreads + tid] += e;
    else far += e;
  };
  if (live) {
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
      for (int i = 0; i < EPV; ++i) add(widen<E>(raw[k], i));
    if (xv > -CUDART_INF_F) add(xv);
  }
  __syncthreads();
  // Slice totals per bin: 4 threads per bin, 64 columns each (rotated so the
  // lanes of a warp hit different banks).
  float* out = L.summ + static_cast<int64_t>(sbase + s) * kSummary;
  {
    const int b = tid >> 2, part = tid & 3;
    float acc = 0.0f;
#pragma unroll 8
    for (int t = 0; t < 64; ++t) acc += ph[b * kSThreads + part * 64 + ((t + 4 * (b & 7) + part) & 63)];
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if (part == 0) out[4 + b] = acc;
  }
  far = block_sum<kSThreads>(far, sh.red_f);
  if (tid == 0) {
    out[0] = ms;
    out[1] = far;
    __threadfence();
    const unsigned prev = atomicAdd(L.counters + grow, 1u);
    sh.last = prev == static_cast<unsigned>(ns - 1);
  }
  __syncthreads();
  if (!sh.last) return;
  __threadfence();

  // 3. Last slice block of the row: merge the summaries.
  const float* sum0 = L.summ + static_cast<int64_t>(sbase) * kSummary;
  float m = -CUDART_INF_F;
  for (int q = tid; q < ns; q += kSThreads) m = fmaxf(m, __ldcg(sum0 + q * kSummary));
  m = block_max<kSThreads>(m, sh.red_f);
  const bool empty = !(m > -CUDART_INF_F);
  const float mc = m * c;
  uint32_t tau = 0u;
  int32_t cut = INT32_MAX;
  double K = 0.0;
  if (!empty) {
    const int G = half_octave(m, c);
    // Warp w merges slices w, w+8, ...; each lane holds bins lane, lane+32.
    float b0 = 0.0f, b1 = 0.0f, fsum = 0.0f;
    for (int q = warp; q < ns; q += kWarps) {
      const float* sq = sum0 + q * kSummary;
      const float mq = __ldcg(sq);
      if (!(mq > -CUDART_INF_F)) continue;
      const float f = ex2(fmaf(mq, c, -mc));  // 2^((m_q - m) c)
      const int D = G - half_octave(mq, c);
      const int l0 = lane - D, l1 = lane + 32 - D;
      if (l0 >= 0) b0 += __ldcg(sq + 4 + l0) * f;
      if (l1 >= 0) b1 += __ldcg(sq + 4 + l1) * f;
      // Slice bins that fall below the merged window, and the slice's own
      // mass below its bins.
      float below = 0.0f;
      if (lane >= kGB - D) below += __ldcg(sq + 4 + lane);
      if (lane + 32 >= kGB - D) below += __ldcg(sq + 4 + lane + 32);
      below = warp_sum(below);
      fsum += (below + __ldcg(sq + 1)) * f;
    }
    sh.mbins[warp][lane] = b0;
    sh.mbins[warp][lane + 32] = b1;
    if (lane == 0) sh.mfar[warp] = fsum;
    __syncthreads();
    if (warp == 0) {
      double r0 = 0.0, r1 = 0.0, fr = 0.0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        r0 += static_cast<double>(sh.mbins[w][2 * lane]);
        r1 += static_cast<double>(sh.mbins[w][2 * lane + 1]);
        fr += static_cast<double>(sh.mfar[w]);
      }
      const double pair = r0 + r1;
      double incl = pair;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const double tot = __shfl_sync(0xffffffffu, incl, 31) + fr;
      const double lim = static_cast<double>(L.top_p) * tot;
      const double before = incl - pair;
      int hit = -1;
      double a0 = 0.0;
      if (before + r0 > lim) {
        hit = 2 * lane;
        a0 = before;
      } else if (before + pair > lim) {
        hit = 2 * lane + 1;
        a0 = before + r0;
      }
      const unsigned hb = __ballot_sync(0xffffffffu, hit >= 0);
      const int src = hb ? __ffs(hb) - 1 : 0;
      const int bs = hb ? __shfl_sync(0xffffffffu, hit, src) : -1;
      const double a = __shfl_sync(0xffffffffu, a0, src);
      if (lane == 0) {
        sh.total = tot;
        sh.limit = lim;
        sh.gstar = bs;
        sh.above0 = a;
      }
    }
    __syncthreads();
    const int bstar = sh.gstar;
    const double limit = sh.limit, above0 = sh.above0, total = sh.total;
    __syncthreads();
    bool generic = false;
    if (bstar < 0) {
      // Nothing in the window reaches top_p * S: every id is kept, or the cut
      // lies among the masses below the window (exact path).
      generic = limit < total;
      if (!generic) K = total;
    } else {
      generic = !resolve_row<E>(sh, row, S, c, mc, G - bstar, above0, limit, tau, cut, K);
    }
    if (generic) {
      __syncthreads();
      generic_select<E>(sh, row, S, c, mc, L.top_p, tau, cut, K);
    }
  }
  if (tid == 0) {
    RowStats st;
    st.m = m;
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
}

template <typename E>
static sv_status launch_typed(const StatsLaunch& L, cudaStream_t stream) {
  static FuncAttrCache cache;
  auto kern = topp_slice_kernel<E>;
  const size_t smem = sizeof(ToppShared);
  if (!cache.ensure(reinterpret_cast<const void*>(kern), smem, false)) return SV_ERR_CUDA;
  const long long blocks = static_cast<long long>(L.set[0].rows) * L.nslices[0] +
                           (L.nsets > 1 ? static_cast<long long>(L.set[1].rows) * L.nslices[1] : 0);
  if (blocks == 0) return SV_OK;
  if (blocks > INT32_MAX) return SV_ERR_UNSUPPORTED;
  kern<<<static_cast<unsigned>(blocks), kSThreads, smem, stream>>>(L);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  note_launch(stream);
  return SV_OK;
}

int topp_slices(int len) { return len <= 0 ? 1 : (len + kSlice - 1) / kSlice; }

size_t topp_scratch_bytes(int rows0, int len0, int rows1, int len1) {
  const size_t slices = static_cast<size_t>(rows0) * topp_slices(len0) + static_cast<size_t>(rows1) * topp_slices(len1);
  // Slack for the alignment of two separately launched sets.
  return align_up(slices * kSummary * sizeof(float), 256) +
         align_up(static_cast<size_t>(rows0 + rows1) * sizeof(unsigned), 256) + 512;
}

sv_status launch_topp_stats(StatsLaunch L, sv_dtype dtype, void* scratch, cudaStream_t stream) {
  const int rows = L.set[0].rows + (L.nsets > 1 ? L.set[1].rows : 0);
  if (rows == 0) return SV_OK;
  for (int i = 0; i < L.nsets; ++i) L.nslices[i] = topp_slices(L.set[i].len);
  const size_t slices = static_cast<size_t>(L.set[0].rows) * L.nslices[0] +
                        (L.nsets > 1 ? static_cast<size_t>(L.set[1].rows) * L.nslices[1] : 0);
  L.summ = static_cast<float*>(scratch);
  L.counters = reinterpret_cast<unsigned*>(static_cast<char*>(scratch) +
                                           align_up(slices * kSummary * sizeof(float), 256));
  if (cudaMemsetAsync(L.counters, 0, static_cast<size_t>(rows) * sizeof(unsigned), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  return dtype == SV_BF16 ? launch_typed<uint16_t>(L, stream) : launch_typed<float>(L, stream);
}

}  // namespace sv
