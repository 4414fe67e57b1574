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
//  * slice blocks: every block reads one slice of a row (8192 fp32 or 16384
//    bf16 logits, eight 16-byte vectors per thread) into
//    registers and takes the slice maximum.  Each logit falls in the
//    ABSOLUTE eighth-octave bin f = floor(8 * l * c) (c = log2(e)/T), so that
//    bins line up across the slices of a row.  The 256 bins below the slice
//    maximum collect the logits' masses in fixed point relative to the bin's
//    upper edge, v = round(2^F * 2^(l*c - (f+1)/8)) (F = 21 for fp32, 20 for
//    bf16 rows), summed exactly in
//    per-warp u32 histograms (shared-memory integer reductions, no read-
//    modify-write chains); lower logits count in the lowest bin.  Two logits
//    are binned per packed FP32 instruction.  Every logit's bin slot is also
//    stored as one code byte, in logit order.  The block publishes (m_s, top
//    bin, 256 bin sums) and bumps the row's counter;
//  * the row's last slice block merges the summaries (a bin's mass is its
//    summed v times 2^((f+1)/8 - F - m*c) whichever slice it came from),
//    finds the bin f* where the mass from the top first exceeds top_p * S,
//    finds the logits of f* from the code bytes (a quarter of an fp32 row's
//    bytes) and gathers their values, and resolves the cut among them by
//    radix levels over their order keys, ending with an exact sort of the
//    last <= 64 by (logit descending, tie key ascending) walked in double
//    precision.
// Rare rows (the cut in the lowest of the 256 bins under the maximum or
// below, a slice whose lowest bin holds f*, more than 4096 logits in f*)
// rescan the row's values or take an exact radix select over the order keys
// of the row.
#include "sv_rows.cuh"

#include <cuda_bf16.h>

namespace sv {

constexpr int kSThreads = 256;
// Logits per thread per slice (eight 16-byte vectors either way) and the
// fixed-point scale of the slice bins: a warp sums at most 32 * kEPT + 32
// values below kFix, which stays under 2^32.
template <typename E> struct SliceShape;
template <> struct SliceShape<float> {
  static constexpr int kEPT = 32;
  static constexpr int kFixLog2 = 21;
  static constexpr float kFix = 2097152.0f;  // 2^21
};
template <> struct SliceShape<uint16_t> {
  static constexpr int kEPT = 64;
  static constexpr int kFixLog2 = 20;
  static constexpr float kFix = 1048576.0f;  // 2^20
};
constexpr int kMinSlice = kSThreads * 32;       // the smaller slice (scratch sizing)
constexpr int kNB = 256;                        // eighth-octave bins under a slice maximum
constexpr int kSummary = 4 + kNB;               // floats per slice summary
constexpr int kCandCap = 4096;                  // candidates of the cut bin in shared memory
constexpr int kFinal = 64;
constexpr int kMaxStaged = kCandCap / 2;         // slice headers staged in shared memory
constexpr int kRegion = kCandCap / (kSThreads / 32);  // candidates per warp in the rescan
constexpr int kWarps = kSThreads / 32;
constexpr float kFixCand = 524288.0f;           // 2^19: candidate level masses
// Magic constants of the FP32-pipe floor and rounding: x + 1.5 * 2^23 holds
// an integer n in its low mantissa bits for |n| < 2^22 (0x4B400000 + n).
constexpr float kMagicFloor = 12582912.0f;  // 1.5 * 2^23
constexpr uint32_t kMagicFloorBits = 0x4B400000u;
constexpr float kMagicRound = 8388608.0f;   // 2^23: 0x4B000000 + n for n in [0, 2^23)
constexpr uint32_t kMagicRoundBits = 0x4B000000u;
constexpr double kScale40 = 1099511627776.0;    // generic path: masses in units of 2^-40
constexpr double kInv40 = 1.0 / 1099511627776.0;

struct ToppShared {
  union {
    unsigned wh[kWarps][kNB];                   // slice phase: per-warp bin sums (fixed point)
    struct {
      float x[kCandCap];                        // merge phase: candidate logits
      int j[kCandCap];                          //              and their ids
    } cand;
    unsigned gh[4][256];                        // generic path: count and 3 mass limbs
  };
  unsigned hcnt[256];
  unsigned hmass[256];
  unsigned long long tmass[256];
  unsigned tcnt[256];
  double scan[32];
  float red_f[32];
  unsigned long long red_u[32];
  int gidx[kFinal];
  int wcnt[kWarps];
  int last;
  int ncand;
  int sel;
  int found;
  unsigned long long sel_above;
  unsigned sel_cnt;
  int gstar;
  int pick_sec;
  unsigned pick_key;
  double above0, limit, total, kept_mass, unit;
  float xlo, xhi;
};

// L2 eviction priorities: the slice pass reads the logits evict-first (they
// are read again only where a row falls back to the value scan, or for the
// few logits of the cut bin) and writes the code bytes evict-last, so they
// survive until the row's last block reads and drops them.  Hints only:
// results do not depend on them.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void stg_hint(uint32_t* a, uint32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(a), "r"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void stg_hint(uint2* a, uint2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(a), "r"(v.x), "r"(v.y), "l"(pol)
               : "memory");
}
__device__ __forceinline__ uint4 ldg_hint(const uint4* a, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(a), "l"(pol));
  return r;
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

// Two bf16 logits in one 32-bit word.
__device__ __forceinline__ __nv_bfloat162 bf2_of(uint32_t w) {
  __nv_bfloat162 r;
  memcpy(&r, &w, sizeof(r));
  return r;
}

// exp2 that the compiler may not merge with an identical earlier one.
__device__ __forceinline__ float ex2v(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^n for an integer n in the normal double range.
__device__ __forceinline__ double pow2i(int n) {
  return __longlong_as_double(static_cast<long long>(n + 1023) << 52);
}

// 2^(i/8) for i = 0..7, from the binary digits of i.
__device__ __forceinline__ double pow2_eighths(int i) {
  double r = 1.0;
  if (i & 1) r *= 1.0905077326652577;  // 2^(1/8)
  if (i & 2) r *= 1.1892071150027210;  // 2^(1/4)
  if (i & 4) r *= 1.4142135623730951;  // 2^(1/2)
  return r;
}

// Visit every logit of a row (body vectors strided over the block, then the
// scalar head and tail): f(value, index), index -1 for padding.
template <typename E, typename F>
__device__ __forceinline__ void for_row(const E* row, int len, F&& f) {
  constexpr int EPV = Elem<E>::kPerVec;
  const RowSplit rs = split_row(row, len);
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  constexpr int U = 8;
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

// Visit every logit of a row with the loads of the next batch of 16-byte
// vectors issued before the current batch is used; f(value, index), index -1
// for padding.  Block-uniform trip counts (f may use full-warp votes).
template <typename E, typename F>
__device__ __forceinline__ void scan_row(const E* row, int len, F&& f) {
  constexpr int EPV = Elem<E>::kPerVec;
  constexpr int U = 4;
  constexpr int kStep = kSThreads * U;
  const RowSplit rs = split_row(row, len);
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  const int v0 = static_cast<int>(threadIdx.x);
  const uint64_t drop = l2_policy_evict_first();
  auto load = [&](uint4* w, int base) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = base + v0 + u * kSThreads;
      w[u] = v < rs.nvec ? ldg_hint(vp + v, drop) : Elem<E>::neg_inf_vec();
    }
  };
  auto use = [&](const uint4* w, int base) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = base + v0 + u * kSThreads;
#pragma unroll
      for (int i = 0; i < EPV; ++i) f(Elem<E>::at(w[u], i), v < rs.nvec ? rs.head + v * EPV + i : -1);
    }
  };
  uint4 a[U], b[U];
#pragma unroll
  for (int u = 0; u < U; ++u) b[u] = Elem<E>::neg_inf_vec();
  if (rs.nvec > 0) load(a, 0);
  // One copy of the loop body: the next batch lands in b, then moves to a.
  for (int base = 0; base < rs.nvec; base += kStep) {
    if (base + kStep < rs.nvec) load(b, base + kStep);
    use(a, base);
#pragma unroll
    for (int u = 0; u < U; ++u) a[u] = b[u];
  }
  const int ntail = len - rs.tail0;
  for (int t0 = 0; t0 < rs.head + ntail; t0 += kSThreads) {
    const int t = t0 + static_cast<int>(threadIdx.x);
    const int j = t < rs.head ? t : (t < rs.head + ntail ? rs.tail0 + (t - rs.head) : -1);
    f(j >= 0 ? Elem<E>::load(row + j) : -CUDART_INF_F, j);
  }
}

// The smallest float x with floor(x * c8) >= b (c8 > 0): x * c8 rounds
// monotonically, so the logits with floor(x * c8) == b are exactly
// [first_at_or_above(b), first_at_or_above(b + 1)).
__device__ __forceinline__ float first_at_or_above(float b, float c8) {
  float x = b / c8;
  for (int i = 0; i < 64 && x * c8 >= b; ++i) x = nextafterf(x, -CUDART_INF_F);
  for (int i = 0; i < 64 && x * c8 < b; ++i) x = nextafterf(x, CUDART_INF_F);
  return x;
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
  unsigned* h = &sh.gh[0][0];  // [count, m0, m1, m2][256]
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

// Ids of the logits in [xlo, xhi) into this warp's region of sh.cand.j:
// per batch of 16-byte vectors each thread builds a bit mask of its
// candidates, then the warp drains the set bits with ballots (the values
// are fetched afterwards).  Returns the warp's count, which may exceed the
// region (entries past it are dropped).  Block-uniform trip counts.
template <typename E>
__device__ __forceinline__ int collect_ids(ToppShared& sh, const E* row, int len, float xlo, float xhi) {
  constexpr int EPV = Elem<E>::kPerVec;
  constexpr int U = 4;
  constexpr int kStep = kSThreads * U;
  static_assert(U * EPV <= 32, "one mask bit per logit of a batch");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lane_lt = (1u << lane) - 1u;
  int* region = sh.cand.j + warp * kRegion;
  const RowSplit rs = split_row(row, len);
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  const uint64_t drop = l2_policy_evict_first();
  const int v0 = static_cast<int>(threadIdx.x);
  int wn = 0;
  auto load = [&](uint4* w, int base) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = base + v0 + u * kSThreads;
      w[u] = v < rs.nvec ? ldg_hint(vp + v, drop) : Elem<E>::neg_inf_vec();
    }
  };
  auto use = [&](const uint4* w, int base) {
    unsigned mask = 0;
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < EPV; ++i) {
        const float x = Elem<E>::at(w[u], i);
        if (x >= xlo && x < xhi) mask |= 1u << (u * EPV + i);
      }
    while (__ballot_sync(0xffffffffu, mask != 0)) {
      const bool has = mask != 0;
      const unsigned bal = __ballot_sync(0xffffffffu, has);
      if (has) {
        const int bit = __ffs(mask) - 1;
        const int u = bit / EPV, i = bit - u * EPV;
        const int slot = wn + __popc(bal & lane_lt);
        if (slot < kRegion) region[slot] = rs.head + (base + v0 + u * kSThreads) * EPV + i;
        mask &= mask - 1;
      }
      wn += __popc(bal);
    }
  };
  uint4 a[U], b[U];
#pragma unroll
  for (int u = 0; u < U; ++u) b[u] = Elem<E>::neg_inf_vec();
  if (rs.nvec > 0) load(a, 0);
  for (int base = 0; base < rs.nvec; base += kStep) {
    if (base + kStep < rs.nvec) load(b, base + kStep);
    use(a, base);
#pragma unroll
    for (int u = 0; u < U; ++u) a[u] = b[u];
  }
  const int ntail = len - rs.tail0;
  for (int t0 = 0; t0 < rs.head + ntail; t0 += kSThreads) {
    const int t = t0 + static_cast<int>(threadIdx.x);
    const int j = t < rs.head ? t : (t < rs.head + ntail ? rs.tail0 + (t - rs.head) : -1);
    const float x = j >= 0 ? Elem<E>::load(row + j) : -CUDART_INF_F;
    const bool cand = x >= xlo && x < xhi;
    const unsigned bal = __ballot_sync(0xffffffffu, cand);
    const int slot = wn + __popc(bal & lane_lt);
    if (cand && slot < kRegion) region[slot] = j;
    wn += __popc(bal);
  }
  return wn;
}

// Ids of the logits of the cut bin into this warp's region of sh.cand.j,
// found by the slices' code bytes instead of their values: in slice q the
// logits of the cut bin are those of bin slot tq[q] (>= 0; -1: the slice has
// none; every slice's cut bin lies above its lowest bin), whose code byte is
// tq[q] + 1.  Sixteen
// codes per 16-byte load, four compared at once (a byte of w ^ t is zero
// exactly where the code matches); the scalar head and tail logits are
// compared by value.  The codes are dropped from L2 afterwards (they are
// never needed again).  Returns the warp's count, which may exceed the
// region (entries past it are dropped).  Block-wide.
template <typename E>
__device__ __forceinline__ int collect_codes(ToppShared& sh, const uint8_t* codes, const int* tq, int ns,
                                             const E* row, int len, float xlo, float xhi) {
  constexpr int SL = SliceShape<E>::kEPT * kSThreads;  // logits (code bytes) per slice
  constexpr int Q16 = SL / 16;                           // 16-byte code vectors per slice
  static_assert((Q16 & (Q16 - 1)) == 0, "slices of a power-of-two size");
  constexpr int kQShift = Q16 == 512 ? 9 : 10;
  static_assert((1 << kQShift) == Q16, "shift of the slice index");
  constexpr int U = 2;  // code vectors per thread per batch
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* region = sh.cand.j + warp * kRegion;
  const RowSplit rs = split_row(row, len);
  const uint4* c4 = reinterpret_cast<const uint4*>(codes);
  const int total = ns * Q16;
  int wn = 0;
  uint4 na[U];
  int nt[U];
  auto load = [&](int g0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = g0 + u * kSThreads + tid;
      nt[u] = g < total ? tq[g >> kQShift] : -1;
      na[u] = nt[u] >= 0 ? __ldcg(c4 + g) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load(0);
  for (int g0 = 0; g0 < total; g0 += U * kSThreads) {
    uint4 cv[U];
    int t[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      cv[u] = na[u];
      t[u] = nt[u];
    }
    if (g0 + U * kSThreads < total) load(g0 + U * kSThreads);
    // Zero-byte masks of w ^ t (the top bit of each matching byte), folded
    // into one bit per code of the batch: word i's mask shifted right by
    // 7 - i puts the match of its byte b at bit 8b + i, so vector u's four
    // words fill bits 32u + 8b + i (code 4i + b of the vector).  A vector of
    // a slice without the cut bin is zero and is compared with code 1.
    unsigned long long bm = 0ull;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t t4 = t[u] >= 0 ? static_cast<uint32_t>(t[u] + 1) * 0x01010101u : 0x01010101u;
      const uint32_t w[4] = {cv[u].x, cv[u].y, cv[u].z, cv[u].w};
      uint32_t vm = 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x4 = w[i] ^ t4;
        vm |= ~(((x4 & 0x7f7f7f7fu) + 0x7f7f7f7fu) | x4 | 0x7f7f7f7fu) >> (7 - i);
      }
      bm |= static_cast<unsigned long long>(vm) << (32 * u);
    }
    const int cnt = __popcll(bm);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int slot = wn + incl - cnt;
    // One loop over the set bits (its trip count is the lane's count, not
    // one loop per word).
    while (bm) {
      const int k = __ffsll(static_cast<long long>(bm)) - 1;
      bm &= bm - 1;
      const int g = g0 + (k >> 5) * kSThreads + tid;
      const int q = g >> kQShift;
      const int e = 4 * (k & 7) + ((k >> 3) & 3);  // code of the vector
      if (slot < kRegion) region[slot] = rs.head + q * SL + (g & (Q16 - 1)) * 16 + e;
      ++slot;
    }
    wn += __shfl_sync(0xffffffffu, incl, 31);
  }
  // The scalar head and tail logits, by value.
  const unsigned lane_lt = (1u << lane) - 1u;
  const int ntail = len - rs.tail0;
  for (int t0 = 0; t0 < rs.head + ntail; t0 += kSThreads) {
    const int t = t0 + tid;
    const int j = t < rs.head ? t : (t < rs.head + ntail ? rs.tail0 + (t - rs.head) : -1);
    const float x = j >= 0 ? Elem<E>::load(row + j) : -CUDART_INF_F;
    const bool cand = x >= xlo && x < xhi;
    const unsigned bal = __ballot_sync(0xffffffffu, cand);
    const int slot = wn + __popc(bal & lane_lt);
    if (cand && slot < kRegion) region[slot] = j;
    wn += __popc(bal);
  }
  // Drop the codes from L2 without writing them back (128-byte lines; every
  // slice's codes start on a 128-byte boundary), once every warp has read
  // them.
  __syncthreads();
  for (int i = tid; i < total / 8; i += kSThreads)
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(c4 + 8 * i) : "memory");
  return wn;
}

// The cut among the candidates of the cut bin (n <= kCandCap, in
// sh.cand): radix levels over their order keys, each keeping the digit where
// the mass from the top first exceeds the limit (counts and fixed-point
// masses v = round(2^19 * 2^(l*c + nb)), nb = -(f*+1)/8), then an exact sort
// of the last <= 64 walked in double precision, or for a larger group of
// equal logits a cut by tie key.  above0 and limit are masses relative to the
// row maximum; `unit` is the mass of one fixed-point unit.  Every
// candidate's order key lies in [klo, khi] (the cut bin's key range).
template <typename E>
__device__ void resolve_candidates(ToppShared& sh, const RowSet& S, float c, float mc, int n, float nb,
                                   double above0, double limit, double unit, uint32_t klo, uint32_t khi,
                                   uint32_t& tau, int32_t& cut, double& K) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned long long above_f = 0;
  uint32_t kbase = 0;
  int cnt = n;
  if (n > kFinal) {
    const uint32_t kmin = klo, kmax = khi;
    const double lim_rel = limit - above0;
    const unsigned long long lim_f = lim_rel > 0.0 ? static_cast<unsigned long long>(lim_rel / unit) : 0ull;
    kbase = kmin;
    const uint32_t span = kmax - kmin;
    int shift = span ? max(0, 32 - __clz(static_cast<int>(span)) - 8) : 0;
#pragma unroll 1
    for (;;) {
      for (int t = tid; t < 256; t += kSThreads) {
        sh.hcnt[t] = 0u;
        sh.hmass[t] = 0u;
      }
      __syncthreads();
      for (int i = tid; i < cnt; i += kSThreads) {
        const float x = sh.cand.x[i];
        const uint32_t d = min((order_key(x) - kbase) >> shift, 255u);  // < 256 for keys in range
        atomicAdd(&sh.hcnt[d], 1u);
        atomicAdd(&sh.hmass[d], __float2uint_rn(ex2v(fmaf(x, c, nb)) * kFixCand));
      }
      __syncthreads();
      for (int t = tid; t < 256; t += kSThreads) {
        sh.tcnt[t] = sh.hcnt[t];
        sh.tmass[t] = sh.hmass[t];
      }
      __syncthreads();
      crossing_desc(sh, 255, above_f, lim_f);
      __syncthreads();
      const uint32_t dsel = static_cast<uint32_t>(sh.sel);
      above_f = sh.sel_above;
      // Keep the candidates of digit dsel, in order, in place: chunks of four
      // entries per thread, each read completely before any of it is written.
      int kept_n = 0;
      for (int b0 = 0; b0 < cnt; b0 += 4 * kSThreads) {
        float xv[4];
        int jv[4];
        unsigned km = 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int i = b0 + 4 * tid + r;
          xv[r] = 0.0f;
          jv[r] = 0;
          if (i < cnt) {
            xv[r] = sh.cand.x[i];
            jv[r] = sh.cand.j[i];
            if (((order_key(xv[r]) - kbase) >> shift) == dsel) km |= 1u << r;
          }
        }
        const int k = __popc(km);
        int incl = k;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane == 31) sh.wcnt[warp] = incl;
        __syncthreads();
        int off = kept_n + incl - k, chunk = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const int nw = sh.wcnt[w];
          if (w < warp) off += nw;
          chunk += nw;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (km & (1u << r)) {
            sh.cand.x[off] = xv[r];
            sh.cand.j[off] = jv[r];
            ++off;
          }
        }
        kept_n += chunk;
        __syncthreads();
      }
      cnt = kept_n;
      kbase += dsel << shift;
      if (cnt <= kFinal || shift == 0) break;
      shift = max(0, shift - 8);
    }
  }
  const double above = above0 + static_cast<double>(above_f) * unit;
  if (cnt <= kFinal) {
    // Sort the final group by (logit descending, tie key ascending), walk it.
    if (warp == 0) {
      unsigned long long a = 0, b = 0;
      if (lane < cnt)
        a = (static_cast<unsigned long long>(order_key(sh.cand.x[lane])) << 32) |
            (0xffffffffu - static_cast<uint32_t>(tie_key(S, sh.cand.j[lane])));
      if (lane + 32 < cnt)
        b = (static_cast<unsigned long long>(order_key(sh.cand.x[lane + 32])) << 32) |
            (0xffffffffu - static_cast<uint32_t>(tie_key(S, sh.cand.j[lane + 32])));
      int ra = 0, rb = 0;
#pragma unroll 4
      for (int j2 = 0; j2 < 32; ++j2) {
        const unsigned long long xa2 = __shfl_sync(0xffffffffu, a, j2);
        const unsigned long long xb2 = __shfl_sync(0xffffffffu, b, j2);
        ra += (xa2 > a) + (xb2 > a);
        rb += (xa2 > b) + (xb2 > b);
      }
      if (lane < cnt) sh.gidx[ra] = lane;
      if (lane + 32 < cnt) sh.gidx[rb] = lane + 32;
      __syncwarp();
      // Masses in sorted order (lane r: ranks r and r + 32), prefix sums in
      // double, the first rank whose inclusive mass exceeds the limit.
      double i0 = lane < cnt ? static_cast<double>(weight(sh.cand.x[sh.gidx[lane]], c, mc)) : 0.0;
      double i1 = lane + 32 < cnt ? static_cast<double>(weight(sh.cand.x[sh.gidx[lane + 32]], c, mc)) : 0.0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double y0 = __shfl_up_sync(0xffffffffu, i0, o);
        const double y1 = __shfl_up_sync(0xffffffffu, i1, o);
        if (lane >= o) {
          i0 += y0;
          i1 += y1;
        }
      }
      i1 += __shfl_sync(0xffffffffu, i0, 31);
      const unsigned h0 = __ballot_sync(0xffffffffu, lane < cnt && above + i0 > limit);
      const unsigned h1 = __ballot_sync(0xffffffffu, lane + 32 < cnt && above + i1 > limit);
      const int pick = h0 ? __ffs(h0) - 1 : (h1 ? 31 + __ffs(h1) : cnt - 1);
      const double ip0 = __shfl_sync(0xffffffffu, i0, pick & 31);
      const double ip1 = __shfl_sync(0xffffffffu, i1, pick & 31);
      if (lane == 0) {
        const int ip = sh.gidx[pick];
        sh.pick_key = order_key(sh.cand.x[ip]);
        sh.pick_sec = tie_key(S, sh.cand.j[ip]);
        sh.kept_mass = above + (pick < 32 ? ip0 : ip1);
      }
    }
    __syncthreads();
    tau = sh.pick_key;
    cut = sh.pick_sec;
    K = sh.kept_mass;
    return;
  }
  // More than 64 equal logits at the cut: keep the nk with the lowest tie keys.
  const double e_g = static_cast<double>(weight(sh.cand.x[0], c, mc));
  double nkd = floor((limit - above) / e_g) + 1.0;
  if (!(nkd >= 1.0)) nkd = 1.0;
  const unsigned nk = nkd >= static_cast<double>(cnt) ? static_cast<unsigned>(cnt) : static_cast<unsigned>(nkd);
  tau = kbase;
  K = above + static_cast<double>(nk) * e_g;
  cut = INT32_MAX;
  if (nk < static_cast<unsigned>(cnt)) {
    uint32_t sp = 0;
    unsigned need = nk;
#pragma unroll 1
    for (int q = 0; q < 3; ++q) {
      const int sb = 16 - 8 * q;
      for (int t = tid; t < 256; t += kSThreads) sh.hcnt[t] = 0u;
      __syncthreads();
      for (int s = tid; s < cnt; s += kSThreads) {
        const uint32_t s2 = static_cast<uint32_t>(tie_key(S, sh.cand.j[s]));
        if (q == 0 || (s2 >> (sb + 8)) == sp) atomicAdd(&sh.hcnt[(s2 >> sb) & 255], 1u);
      }
      __syncthreads();
      for (int t = tid; t < 256; t += kSThreads) sh.tcnt[t] = sh.hcnt[t];
      __syncthreads();
      crossing_count(sh, need);
      __syncthreads();
      sp = (sp << 8) | static_cast<uint32_t>(sh.sel);
      need -= static_cast<unsigned>(sh.sel_above);
      __syncthreads();
    }
    cut = static_cast<int32_t>(sp);
  }
}

// Bin every logit of this thread's vectors with add (which returns the
// logit's code, (bin slot + 1) mod 256) and store the codes as bytes in
// logit order: vector k of thread tid holds logits
// (k * kSThreads + tid) * EPV + 0..EPV-1 of the slice.
template <typename E, int VPT, typename F>
__device__ __forceinline__ void bin_vectors(const uint4 (&raw)[VPT], uint8_t* codes, F&& add) {
  constexpr int EPV = Elem<E>::kPerVec;
  const int tid = threadIdx.x;
  const uint64_t keep = l2_policy_evict_last();
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    uint32_t w[EPV / 4];
#pragma unroll
    for (int h = 0; h < EPV / 4; ++h) {
      w[h] = 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) w[h] |= add(Elem<E>::at(raw[k], 4 * h + j)) << (8 * j);
    }
    if constexpr (EPV == 4) {
      stg_hint(reinterpret_cast<uint32_t*>(codes) + k * kSThreads + tid, w[0], keep);
    } else {
      stg_hint(reinterpret_cast<uint2*>(codes) + k * kSThreads + tid, make_uint2(w[0], w[1]), keep);
    }
  }
}

// Binning of two logits at once with the packed FP32 instructions of sm_100
// and later (two lanes per instruction), for the fast path of the slice
// pass; bit for bit the scalar binning.  With y = l * c8 and fy = floor(y):
// E = (2^23 + 1 + Gs) + (-y) rounded up is 2^23 + 1 + (Gs - fy) exactly (the
// sum lies in [2^23, 2^24), where the spacing is 1, for every logit of the
// slice), so the mantissa of E holds 1 + Gs - fy; clamped as an integer at
// 1 + 255 it gives the bin idx = min(Gs - fy, 255) + 1 and the clamped floor
// fy_c.  Then -(fy_c + 1)/8 = (E_c - 2^23 - 2 - Gs)/8 (exact), t = l*c plus
// that in one rounding, and v = round(2^F * 2^t) by the magic addition.
// The low byte of E_c is the logit's code, (idx + 1) mod 256.
struct PairBins {
  uint64_t nc8;    // (-c8, -c8)
  uint64_t mg;     // (2^23 + 1 + Gs, ...)
  uint64_t kg;     // (-(2^23 + 2 + Gs) / 8, ...)
  uint64_t c;      // (c, c)
  uint64_t fix;    // (2^F, 2^F)
};
constexpr uint32_t kPairBitsIdx0 = 0x4B000001u;  // bits of E_c for idx = 0

__device__ __forceinline__ uint64_t pair_of(float a, float b) {
  return static_cast<uint64_t>(__float_as_uint(a)) | (static_cast<uint64_t>(__float_as_uint(b)) << 32);
}

// (E_c bits, v) of the logits x = (x0, x1) packed low/high.
__device__ __forceinline__ void bin_pair(uint64_t x, const PairBins& k, uint32_t& e0, uint32_t& e1, uint32_t& v0,
                                         uint32_t& v1) {
  uint64_t e;
  asm("{\n\t.reg .b64 y;\n\t"
      "mul.rn.f32x2 y, %1, %2;\n\t"
      "add.rp.f32x2 %0, y, %3;\n\t"
      "}"
      : "=l"(e)
      : "l"(x), "l"(k.nc8), "l"(k.mg));
  e0 = min(static_cast<uint32_t>(e), kPairBitsIdx0 + 255u);
  e1 = min(static_cast<uint32_t>(e >> 32), kPairBitsIdx0 + 255u);
  const uint64_t ec = static_cast<uint64_t>(e0) | (static_cast<uint64_t>(e1) << 32);
  uint64_t t;
  asm("{\n\t.reg .b64 g;\n\t"
      "fma.rn.f32x2 g, %1, %5, %2;\n\t"
      "fma.rn.f32x2 %0, %3, %4, g;\n\t"
      "}"
      : "=l"(t)
      : "l"(ec), "l"(k.kg), "l"(x), "l"(k.c), "l"(0x3E0000003E000000ull));  // (1/8, 1/8)
  const float p0 = ex2(__uint_as_float(static_cast<uint32_t>(t)));
  const float p1 = ex2(__uint_as_float(static_cast<uint32_t>(t >> 32)));
  uint64_t w;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(w) : "l"(pair_of(p0, p1)), "l"(k.fix), "l"(0x4B0000004B000000ull));
  v0 = static_cast<uint32_t>(w) - kMagicRoundBits;
  v1 = static_cast<uint32_t>(w >> 32) - kMagicRoundBits;
}

// The slice's vectors through bin_pair: bin sums by shared-memory integer
// reductions at whs_adj + 4 * E_c (whs_adj = the warp histogram's address
// less 4 * kPairBitsIdx0), and the codes as bytes in logit order, as
// bin_vectors stores them.
template <typename E, int VPT>
__device__ __forceinline__ void bin_vectors_x2(const uint4 (&raw)[VPT], uint8_t* codes, const PairBins& k,
                                               uint32_t whs_adj) {
  constexpr int EPV = Elem<E>::kPerVec;
  const int tid = threadIdx.x;
  const uint64_t keep = l2_policy_evict_last();
#pragma unroll
  for (int q = 0; q < VPT; ++q) {
    const uint32_t wd[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
    uint32_t word[EPV / 4];
#pragma unroll
    for (int h = 0; h < EPV / 4; ++h) {
      uint32_t eb[4];
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        uint64_t x;
        if constexpr (EPV == 4) {
          x = static_cast<uint64_t>(wd[2 * pr]) | (static_cast<uint64_t>(wd[2 * pr + 1]) << 32);
        } else {
          const uint32_t w2 = wd[2 * h + pr];
          x = static_cast<uint64_t>(w2 << 16) | (static_cast<uint64_t>(w2 & 0xffff0000u) << 32);
        }
        uint32_t v0, v1;
        bin_pair(x, k, eb[2 * pr], eb[2 * pr + 1], v0, v1);
        asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(whs_adj + (eb[2 * pr] << 2)), "r"(v0) : "memory");
        asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(whs_adj + (eb[2 * pr + 1] << 2)), "r"(v1) : "memory");
      }
      word[h] = __byte_perm(__byte_perm(eb[0], eb[1], 0x0040), __byte_perm(eb[2], eb[3], 0x0040), 0x5410);
    }
    if constexpr (EPV == 4) {
      stg_hint(reinterpret_cast<uint32_t*>(codes) + q * kSThreads + tid, word[0], keep);
    } else {
      stg_hint(reinterpret_cast<uint2*>(codes) + q * kSThreads + tid, make_uint2(word[0], word[1]), keep);
    }
  }
}

template <typename E>
__global__ void __launch_bounds__(kSThreads, 5) topp_slice_kernel(StatsLaunch L) {
  constexpr int EPV = Elem<E>::kPerVec;
  constexpr int VPT = SliceShape<E>::kEPT / EPV;  // 16-byte vectors per thread
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
  const float c8 = c * 8.0f;  // 8 * (l * c) == l * c8 exactly

  // Per-warp bin sums start at zero (visible after the barriers of block_max).
#pragma unroll
  for (int i = 0; i < kWarps * kNB / kSThreads; ++i) (&sh.wh[0][0])[i * kSThreads + tid] = 0u;

  // 1. The slice in registers; slice maximum.
  const RowSplit rs = split_row(row, S.len);
  const uint4* vp = reinterpret_cast<const uint4*>(row + rs.head);
  const uint64_t once = l2_policy_evict_first();
  uint4 raw[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = s * VPS + k * kSThreads + tid;
    raw[k] = v < rs.nvec ? ldg_hint(vp + v, once) : Elem<E>::neg_inf_vec();
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
  if constexpr (sizeof(E) == 2) {
    // Packed bf16 maxima, two logits per instruction.
    __nv_bfloat162 m2 = bf2_of(0xff80ff80u);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      m2 = __hmax2(m2, bf2_of(raw[k].x));
      m2 = __hmax2(m2, bf2_of(raw[k].y));
      m2 = __hmax2(m2, bf2_of(raw[k].z));
      m2 = __hmax2(m2, bf2_of(raw[k].w));
    }
    lm = fmaxf(lm, fmaxf(__low2float(m2), __high2float(m2)));
  } else {
    // Three-input maxima (sm_100 and later), two logits per instruction.
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
      for (int i = 0; i < EPV; i += 2) {
        asm("max.f32 %0, %0, %1, %2;" : "+f"(lm) : "f"(Elem<E>::at(raw[k], i)), "f"(Elem<E>::at(raw[k], i + 1)));
      }
  }
  const float ms = block_max<kSThreads>(lm, sh.red_f);

  // 2. Bin sums over the 256 eighth-octaves under the slice maximum.  Lower
  // logits are counted in the lowest bin with their mass relative to its
  // edge (they round to 0 more than 21 octaves below it, and are skipped);
  // the merge never resolves a cut inside that bin (exact path instead).
  // Every logit's bin t = Gs - fy (255: the lowest bin or below) also goes
  // to this slice's code bytes, in the order of the logits.
  uint8_t* codes = L.codes + static_cast<int64_t>(sbase + s) * (VPS * EPV);
  const bool live = ms > -CUDART_INF_F;
  const float Gsf = live ? floorf(ms * c8) : 0.0f;
  const float bottom = Gsf - static_cast<float>(kNB - 1);
  unsigned* wh = sh.wh[warp];
  if (live && fabsf(Gsf) < 4.0e6f) {
    // |floor(l * c8)| < 2^22 across the window: the floor and the rounding to
    // an integer by magic additions in the FP32 pipe (no conversion
    // instruction); fy = max(floor(l * c8), bottom) and the bin Gs - fy come
    // out of the mantissa bits.
    const uint32_t whs = static_cast<uint32_t>(__cvta_generic_to_shared(wh));
    const float gm = Gsf + kMagicFloor;
    auto add = [&](float x) -> uint32_t {
      const float fy = fmaxf(__fadd_rd(x * c8, kMagicFloor) - kMagicFloor, bottom);
      // l*c - (f+1)/8 (in [-1/8, 0] inside the window): the mass relative to
      // the bin's upper edge.
      const float t = fmaf(x, c, fmaf(fy, -0.125f, -0.125f));
      const uint32_t v = __float_as_uint(fmaf(ex2(t), SliceShape<E>::kFix, kMagicRound)) - kMagicRoundBits;
      const uint32_t idx = __float_as_uint(gm - fy) - kMagicFloorBits;
      asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(whs + idx * 4u), "r"(v) : "memory");
      return idx;
    };
    PairBins pk;
    pk.nc8 = pair_of(-c8, -c8);
    const float mg = kMagicRound + 1.0f + Gsf;  // exact: |Gs| < 2^22
    pk.mg = pair_of(mg, mg);
    const float kg = -(kMagicRound + 2.0f + Gsf) * 0.125f;
    pk.kg = pair_of(kg, kg);
    pk.c = pair_of(c, c);
    pk.fix = pair_of(SliceShape<E>::kFix, SliceShape<E>::kFix);
    bin_vectors_x2<E, VPT>(raw, codes, pk, whs - (kPairBitsIdx0 << 2));
    if (xv > -CUDART_INF_F) add(xv);
  } else if (live) {
    // Logits too large for the magic additions: the same bins by floorf and
    // conversions.
    auto add = [&](float x) -> uint32_t {
      const float fy = fmaxf(floorf(x * c8), bottom);
      const float t = fmaf(x, c, fmaf(fy, -0.125f, -0.125f));
      const unsigned v = __float2uint_rn(ex2(t) * SliceShape<E>::kFix);
      const int idx = static_cast<int>(Gsf - fy);
      if (v) atomicAdd(&wh[idx], v);
      return static_cast<uint32_t>(idx + 1) & 0xffu;  // the code
    };
    bin_vectors<E, VPT>(raw, codes, add);
    if (xv > -CUDART_INF_F) add(xv);
  }
  __syncthreads();
  // Publish: slot t holds bin Gs - t.
  float* out = L.summ + static_cast<int64_t>(sbase + s) * kSummary;
  if (tid < kNB) {
    unsigned long long a = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) a += sh.wh[w][tid];
    out[4 + tid] = static_cast<float>(a);
  }
  if (tid == 0) {
    out[0] = ms;
    out[1] = 0.0f;  // no mass outside the bins
    out[2] = Gsf;
    out[3] = 0.0f;
  }
  // One fence on each side, by the thread that counts the slice: the barrier
  // orders the block's summary writes before the releasing fence, and the
  // row's last block reads the other summaries after the acquiring fence
  // and the barrier.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const bool last = atomicAdd(L.counters + grow, 1u) == static_cast<unsigned>(ns - 1);
    if (last) __threadfence();
    sh.last = last;
  }
  __syncthreads();
  if (!sh.last) return;

  // 3. Last slice block of the row: merge the summaries.  Thread b owns the
  // row bin Gr - b; slice bins below the row's 256 go to `far`.
  const float* sum0 = L.summ + static_cast<int64_t>(sbase) * kSummary;
  // The row's slice summaries land in shared memory (one round of
  // asynchronous copies; they span the candidate arrays, free until the
  // candidates are collected) when they fit; else they are read through L2,
  // the slice maxima and top bins staged in shared memory.
  float* ss = reinterpret_cast<float*>(&sh.cand);
  const bool in_smem = ns * kSummary <= 2 * kCandCap;
  if (in_smem) {
    const int n16 = ns * (kSummary / 4);
    for (int i = tid; i < n16; i += kSThreads) cp_async16(ss + 4 * i, sum0 + 4 * i);
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
  }
  auto ldsum = [&](int64_t i) -> float { return in_smem ? ss[i] : __ldcg(sum0 + i); };
  const bool staged = !in_smem && ns <= kMaxStaged;
  float* hm = sh.cand.x;               // slice maximum
  float* hg = sh.cand.x + kMaxStaged;  // slice top bin
  float m = -CUDART_INF_F;
  for (int q = tid; q < ns; q += kSThreads) {
    const float mq = ldsum(static_cast<int64_t>(q) * kSummary);
    m = fmaxf(m, mq);
    if (staged) {
      hm[q] = mq;
      hg[q] = __ldcg(sum0 + static_cast<int64_t>(q) * kSummary + 2);
    }
  }
  m = block_max<kSThreads>(m, sh.red_f);  // its barriers also publish the staging
  const bool empty = !(m > -CUDART_INF_F);
  const float mc = m * c;
  uint32_t tau = 0u;
  int32_t cut = INT32_MAX;
  double K = 0.0;
  if (!empty) {
    const float Grf = floorf(m * c8);
    constexpr float kFixL2 = static_cast<float>(SliceShape<E>::kFixLog2);
    unsigned long long acc = 0;
    float farp = 0.0f;  // slice bins below the row's 256 bins
    if (staged) {
      // Eight slices at a time, every bin load issued before any is used.
#pragma unroll 1
      for (int q0 = 0; q0 < ns; q0 += 8) {
        float v[8], w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int q = q0 + u;
          const bool lq = q < ns && hm[q] > -CUDART_INF_F;
          const int D = lq ? static_cast<int>(Grf - hg[q]) : (1 << 24);
          const float* sq = sum0 + static_cast<int64_t>(lq ? q : 0) * kSummary + 4;
          v[u] = (tid >= D && tid < kNB) ? __ldcg(sq + (tid - D)) : 0.0f;
          // Slice bin Gq - tid lies below the row's bins.
          w[u] = (lq && tid >= kNB - D && tid < kNB) ? __ldcg(sq + tid) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          acc += static_cast<unsigned long long>(v[u]);
          if (w[u] > 0.0f)
            farp += w[u] * ex2v((hg[q0 + u] - static_cast<float>(tid) + 1.0f) * 0.125f - mc - kFixL2);
        }
      }
    } else {
#pragma unroll 1
      for (int q = 0; q < ns; ++q) {
        const int64_t sq = static_cast<int64_t>(q) * kSummary;
        const float mq = ldsum(sq);
        if (!(mq > -CUDART_INF_F)) continue;
        const float Gq = ldsum(sq + 2);
        const int D = static_cast<int>(Grf - Gq);
        if (tid >= D && tid < kNB) acc += static_cast<unsigned long long>(ldsum(sq + 4 + (tid - D)));
        if (tid >= kNB - D && tid < kNB)
          farp += ldsum(sq + 4 + tid) * ex2v((Gq - static_cast<float>(tid) + 1.0f) * 0.125f - mc - kFixL2);
      }
    }
    // Mass of one unit of bin Gr - b: 2^((Gr - b + 1)/8 - kFixLog2 - mc), with the
    // exponent split into whole and eighth powers of two.
    const double frac_unit = static_cast<double>(ex2(floorf(mc) - mc));
    const int kb = static_cast<int>(Grf) - tid + 1;
    const int kq = kb >> 3, kr = kb & 7;
    const double scale =
        pow2i(kq - static_cast<int>(floorf(mc)) - SliceShape<E>::kFixLog2) * pow2_eighths(kr) * frac_unit;
    const double mass = static_cast<double>(acc) * scale;
    double tot;
    const double excl = block_exclusive_scan_d<kSThreads>(mass, sh.scan, &tot);
    const double far_all = static_cast<double>(block_sum<kSThreads>(farp, sh.red_f));
    const double Z = tot + far_all;
    const double limit = static_cast<double>(L.top_p) * Z;
    if (tid == 0) sh.gstar = -1;
    __syncthreads();
    if (mass > 0.0 && excl <= limit && excl + mass > limit) {
      sh.gstar = tid;
      sh.above0 = excl;
      sh.unit = scale * pow2i(SliceShape<E>::kFixLog2 - 19);  // candidate masses: units of 2^-19 of the bin's edge
    }
    __syncthreads();
    const int gstar = sh.gstar;
    const double above0 = sh.above0, unit = sh.unit;
    bool generic = false;
    if (gstar < 0) {
      // Nothing in the 256 bins reaches top_p * S: every id is kept, or the
      // cut lies among the masses below them (exact path).
      generic = limit < Z;
      if (!generic) K = Z;
    } else if (gstar == kNB - 1) {
      generic = true;  // the lowest bin also holds the logits below the window
    } else {
      // Rescan: the logits of the cut bin with their ids, each warp into its
      // own region of the list; if a region overflows, again with one
      // shared counter.
      const float Bf = Grf - static_cast<float>(gstar);
      const unsigned lane_lt = (1u << lane) - 1u;
      // floor(l * c8) == Bf exactly for the logits in [xlo, xhi).
      if (tid == 0) {
        sh.xlo = first_at_or_above(Bf, c8);
        sh.xhi = first_at_or_above(Bf + 1.0f, c8);
      }
      // The cut bin as a code of each slice (in hcnt, free until the
      // resolution); a slice whose lowest bin holds the cut bin (or rows of
      // more slices than the table holds) sends the row to the value scan.
      int* tq = reinterpret_cast<int*>(sh.hcnt);
      if (tid == 0) sh.ncand = ns > kNB;
      __syncthreads();
      for (int q = tid; q < ns && q < kNB; q += kSThreads) {
        int t = -1;
        const float mq = staged ? hm[q] : ldsum(static_cast<int64_t>(q) * kSummary);
        if (mq > -CUDART_INF_F) {
          const float Gq = staged ? hg[q] : ldsum(static_cast<int64_t>(q) * kSummary + 2);
          t = gstar - static_cast<int>(Grf - Gq);
          if (t >= kNB - 1) sh.ncand = 1;
        }
        tq[q] = t;
      }
      __syncthreads();
      const float xlo = sh.xlo, xhi = sh.xhi;
      const int wn = sh.ncand ? collect_ids<E>(sh, row, S.len, xlo, xhi)
                              : collect_codes<E>(sh, L.codes + static_cast<int64_t>(sbase) * (VPS * EPV), tq, ns,
                                                 row, S.len, xlo, xhi);
      if (lane == 0) sh.wcnt[warp] = wn;
      __syncthreads();
      int total_c = 0, my_off = 0, over = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const int nw = sh.wcnt[w];
        over |= nw > kRegion;
        if (w < warp) my_off += nw;
        total_c += nw;
      }
      if (!over) {
        // Pack the regions to the front in warp order: every entry is read
        // into registers before any is written.
        constexpr int kPer = kRegion / 32;
        int rj[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int e2 = lane + 32 * k;
          rj[k] = e2 < wn ? sh.cand.j[warp * kRegion + e2] : 0;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int e2 = lane + 32 * k;
          if (e2 < wn) sh.cand.j[my_off + e2] = rj[k];
        }
        if (tid == 0) sh.ncand = total_c;
      } else if (total_c <= kCandCap) {
        if (tid == 0) sh.ncand = 0;
        __syncthreads();
        scan_row<E>(row, S.len, [&](float x, int j) {
          const bool cand = x >= xlo && x < xhi;
          const unsigned bal = __ballot_sync(0xffffffffu, cand);
          if (bal) {
            int base = 0;
            if (lane == 0) base = atomicAdd(&sh.ncand, __popc(bal));
            base = __shfl_sync(0xffffffffu, base, 0);
            const int slot = base + __popc(bal & lane_lt);
            if (cand && slot < kCandCap) {
              sh.cand.x[slot] = x;
              sh.cand.j[slot] = j;
            }
          }
        });
      } else if (tid == 0) {
        sh.ncand = total_c;
      }
      __syncthreads();
      const int n = sh.ncand;
      generic = n == 0 || n > kCandCap;
      if (!generic) {
        // The candidates' logits: one parallel round of loads (served by L2).
        for (int i = tid; i < n; i += kSThreads) {
          const int j = sh.cand.j[i];
          sh.cand.x[i] = sv_in(j, S.len) ? load_at<E>(row, j) : -CUDART_INF_F;
        }
        __syncthreads();
      }
      if (!generic)
        resolve_candidates<E>(sh, S, c, mc, n, -(Bf + 1.0f) * 0.125f, above0, limit, unit, order_key(xlo),
                              order_key(xhi) - 1u, tau, cut, K);
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
    if (q.elem >= 0 && !empty && sv_in(q.elem, S.len)) {
      const float x = Elem<E>::load(row + q.elem);
      if (kept(order_key(x), q.sec, tau, cut)) st.e_query = weight(x, c, mc);
    }
    S.out[r] = st;
  }
  // Warp 0 alone (thread 0 wrote the statistics): count the row for its
  // batch row and, after the batch row's last one, make its decisions.
  if (L.dec.rec && warp == 0) {
    bool last = false;
    if (tid == 0) last = count_row(L.dec, S, r);
    if (__shfl_sync(0xffffffffu, last, 0)) {
      __threadfence();
      const DecideRecord rc = decide_batch(L.dec, r / S.per_group);
      if ((threadIdx.x & 31) == 0) L.dec.rec[r / S.per_group] = rc;
    }
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

static int slices_of(int len, int slice) { return len <= 0 ? 1 : (len + slice - 1) / slice; }
int topp_slices(int len) { return slices_of(len, kMinSlice); }

// Code bytes: one per logit of every slice, slices padded to whole slices.
// An upper bound from the count of kMinSlice-logit slices: two more such
// slices per row cover the rows cut into the larger bf16 slices.
static size_t topp_code_bytes_bound(size_t slices, int rows) {
  return (slices + 2 * static_cast<size_t>(rows)) * static_cast<size_t>(kMinSlice);
}

size_t topp_scratch_bytes(int rows0, int len0, int rows1, int len1) {
  const size_t slices = static_cast<size_t>(rows0) * topp_slices(len0) + static_cast<size_t>(rows1) * topp_slices(len1);
  // Slack for the alignment of two separately launched sets.
  return align_up(slices * kSummary * sizeof(float), 256) + align_up(topp_code_bytes_bound(slices, rows0 + rows1), 256) +
         align_up(static_cast<size_t>(rows0 + rows1) * sizeof(unsigned), 256) + 512;
}

sv_status launch_topp_stats(StatsLaunch L, sv_dtype dtype, void* scratch, cudaStream_t stream) {
  const int rows = L.set[0].rows + (L.nsets > 1 ? L.set[1].rows : 0);
  if (rows == 0) return SV_OK;
  const int slice = kSThreads * (dtype == SV_BF16 ? SliceShape<uint16_t>::kEPT : SliceShape<float>::kEPT);
  for (int i = 0; i < L.nsets; ++i) L.nslices[i] = slices_of(L.set[i].len, slice);
  const size_t slices = static_cast<size_t>(L.set[0].rows) * L.nslices[0] +
                        (L.nsets > 1 ? static_cast<size_t>(L.set[1].rows) * L.nslices[1] : 0);
  L.summ = static_cast<float*>(scratch);
  // The layout for these slices (within topp_scratch_bytes' bound).
  L.codes = reinterpret_cast<uint8_t*>(static_cast<char*>(scratch) + align_up(slices * kSummary * sizeof(float), 256));
  L.counters = reinterpret_cast<unsigned*>(static_cast<char*>(scratch) +
                                           align_up(slices * kSummary * sizeof(float), 256) +
                                           align_up(slices * static_cast<size_t>(slice), 256));
  if (cudaMemsetAsync(L.counters, 0, static_cast<size_t>(rows) * sizeof(unsigned), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  return dtype == SV_BF16 ? launch_typed<uint16_t>(L, stream) : launch_typed<float>(L, stream);
}

}  // namespace sv
