// Device building blocks shared by the row-statistics and decision kernels:
// online softmax statistics, first argmax, warp-distributed top-F lists and
// deterministic warp reductions.
#pragma once

#include <climits>

#include "specv_common.cuh"

namespace specv {

constexpr int kMaxF = 32;
constexpr int kMaxK = 32;  // drafts per row (K + 1 positions)

template <int VW>
struct Soft {  // online (max, sum) with VW partial sums for accuracy
  float m;
  float s[VW];
  __device__ __forceinline__ void init() {
    m = kNegMax;
#pragma unroll
    for (int k = 0; k < VW; ++k) s[k] = 0.f;
  }
  __device__ __forceinline__ void add(const float (&z)[VW], float c) {
    float vm = z[0];
#pragma unroll
    for (int k = 1; k < VW; ++k) vm = fmaxf(vm, z[k]);  // NaN ignored here
    if (vm > m) {
      const float f = ex2((m - vm) * c);
#pragma unroll
      for (int k = 0; k < VW; ++k) s[k] *= f;
      m = vm;
    }
#pragma unroll
    for (int k = 0; k < VW; ++k) s[k] += ex2((z[k] - m) * c);  // NaN -> sum NaN
  }
  __device__ __forceinline__ float total() const {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < VW; ++k) t += s[k];
    return t;
  }
};

__device__ __forceinline__ void soft_merge(float& m, float& s, float m2, float s2, float c) {
  const float M = fmaxf(m, m2);
  s = s * ex2((m - M) * c) + s2 * ex2((m2 - M) * c);
  m = M;
}

struct Arg {  // first argmax
  float best;
  int32_t idx;
  int32_t bad;
  __device__ __forceinline__ void init() {
    best = neg_inf();
    idx = INT_MAX;
    bad = 0;
  }
  template <int VW>
  __device__ __forceinline__ void add(const float (&z)[VW], int32_t base) {
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      bad |= !(z[k] < pos_inf());  // NaN or +inf
      if (z[k] > best) {
        best = z[k];
        idx = base + k;
      }
    }
  }
  __device__ __forceinline__ void merge(float b2, int32_t i2, int32_t bad2) {
    if (b2 > best || (b2 == best && i2 < idx)) {
      best = b2;
      idx = i2;
    }
    bad |= bad2;
  }
};

__device__ __forceinline__ bool key_beats(float av, int32_t ai, float bv, int32_t bi) {
  return av > bv || (av == bv && ai < bi);
}

// Sorted top-F list over a warp (lane f holds entry f); the order is (logit
// descending, index ascending); empty entries are (-inf, INT_MAX).
struct WarpTopF {
  float v;
  int32_t i;
  float tv;  // entry F-1: the admission threshold, same in every lane
  int32_t ti;
  __device__ __forceinline__ void init() {
    v = neg_inf();
    i = INT_MAX;
    tv = neg_inf();
    ti = INT_MAX;
  }
  __device__ __forceinline__ void insert(float cv, int32_t ci, int F, int lane) {
    const bool ahead = lane < F && key_beats(v, i, cv, ci);
    const int pos = __popc(__ballot_sync(0xffffffffu, ahead));
    if (pos >= F) return;
    const float uv = __shfl_up_sync(0xffffffffu, v, 1);
    const int32_t ui = __shfl_up_sync(0xffffffffu, i, 1);
    if (lane > pos && lane < F) {
      v = uv;
      i = ui;
    } else if (lane == pos) {
      v = cv;
      i = ci;
    }
    tv = __shfl_sync(0xffffffffu, v, F - 1);
    ti = __shfl_sync(0xffffffffu, i, F - 1);
  }
};

// Merge n <= 32 sorted lists lv[r][0..F-1] (shared memory) into out[0..F-1];
// lane r follows list r.  Called by one full warp.
__device__ __forceinline__ void merge_lists(const float (*lv)[kMaxF], const int32_t (*li)[kMaxF],
                                            int n, int F, int lane, float* outv, int32_t* outi) {
  int ptr = 0;
  float hv = neg_inf();
  int32_t hi = INT_MAX;
  if (lane < n) {
    hv = lv[lane][0];
    hi = li[lane][0];
  }
  for (int f = 0; f < F; ++f) {
    float bv = hv;
    int32_t bi = hi;
    int bl = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
      if (key_beats(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
        bl = ol;
      }
    }
    if (lane == 0) {
      outv[f] = bv;
      outi[f] = bi;
    }
    if (lane == bl && bi != INT_MAX) {
      ++ptr;
      if (ptr < F) {
        hv = lv[lane][ptr];
        hi = li[lane][ptr];
      } else {
        hv = neg_inf();
        hi = INT_MAX;
      }
    }
  }
}

// (max, sum) of the online-softmax partials of an aligned group of W lanes
// (the whole warp by default): the group max first, then one rescale per lane
// and a plain sum tree (no exponential per tree step).  The result is in every
// lane of the group.  Lanes without data hold (kNegMax, 0).
template <int W = 32>
__device__ __forceinline__ void warp_soft_all(float& m, float& s, float c) {
  float M = m;
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float t = s * ex2((m - M) * c);
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  m = M;
  s = t;
}

// Reductions over aligned groups of W lanes (W = 32: the whole warp), every
// lane of a group ending with the group's result.  All 32 lanes must call.
template <typename T, int W = 32>
__device__ __forceinline__ T warp_max_all(T x) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) x = max(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// ---- float-float ("double-word") arithmetic -------------------------------
// The sums that locate an inverse-CDF draw need more than fp32's 24 bits, and
// this part's FP64 pipe is narrow: a dependent chain of double adds costs
// about a hundred times a chain of fp32 adds.  A value is kept as an
// unevaluated sum hi + lo of two floats with |lo| <= ulp(hi) / 2, built from
// the error-free transformations TwoSum (Knuth, TAOCP vol. 2, 4.2.2),
// FastTwoSum (Dekker 1971) and the fma-based TwoProd; the add and the
// multiply by a float follow the "accurate" double-word algorithms of Joldes,
// Muller and Popescu (ACM TOMS 44(2), 2017), relative error below 2^-44.
// Explicit round-to-nearest intrinsics keep the compiler from contracting or
// reassociating the steps.
struct FF {
  float hi, lo;
};

__device__ __forceinline__ FF ff(float a) { return FF{a, 0.f}; }

__device__ __forceinline__ FF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bv = __fsub_rn(s, a);
  const float av = __fsub_rn(s, bv);
  return FF{s, __fadd_rn(__fsub_rn(a, av), __fsub_rn(b, bv))};
}

__device__ __forceinline__ FF fast_two_sum(float a, float b) {  // |a| >= |b| (or a == 0)
  const float s = __fadd_rn(a, b);
  return FF{s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ FF ff_add(FF x, FF y) {
  const FF s = two_sum(x.hi, y.hi);
  const FF t = two_sum(x.lo, y.lo);
  const FF v = fast_two_sum(s.hi, __fadd_rn(s.lo, t.hi));
  return fast_two_sum(v.hi, __fadd_rn(t.lo, v.lo));
}

__device__ __forceinline__ FF ff_add(FF x, float y) {
  const FF s = two_sum(x.hi, y);
  return fast_two_sum(s.hi, __fadd_rn(x.lo, s.lo));
}

__device__ __forceinline__ FF ff_neg(FF x) { return FF{-x.hi, -x.lo}; }

__device__ __forceinline__ FF ff_mul(FF x, float y) {
  const float p = __fmul_rn(x.hi, y);
  const float e = __fmaf_rn(x.hi, y, -p);  // exact: x.hi * y = p + e
  return fast_two_sum(p, __fmaf_rn(x.lo, y, e));
}

// the exact product of two floats
__device__ __forceinline__ FF ff_mul(float a, float b) {
  const float p = __fmul_rn(a, b);
  return FF{p, __fmaf_rn(a, b, -p)};
}

// x > y for normalised pairs (|lo| <= ulp(hi) / 2)
__device__ __forceinline__ bool ff_gt(FF x, FF y) {
  return x.hi > y.hi || (x.hi == y.hi && x.lo > y.lo);
}

__device__ __forceinline__ FF shfl_xor(FF x, int o) {
  return FF{__shfl_xor_sync(0xffffffffu, x.hi, o), __shfl_xor_sync(0xffffffffu, x.lo, o)};
}

__device__ __forceinline__ FF shfl_up(FF x, int o) {
  return FF{__shfl_up_sync(0xffffffffu, x.hi, o), __shfl_up_sync(0xffffffffu, x.lo, o)};
}

__device__ __forceinline__ FF shfl(FF x, int src) {
  return FF{__shfl_sync(0xffffffffu, x.hi, src), __shfl_sync(0xffffffffu, x.lo, src)};
}

template <int W = 32>
__device__ __forceinline__ FF warp_ffsum_all(FF x) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) x = ff_add(x, shfl_xor(x, o));
  return x;
}

// inclusive prefix sum over the warp's lanes (Hillis-Steele)
__device__ __forceinline__ FF warp_ffscan(FF x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const FF y = shfl_up(x, o);
    if (lane >= o) x = ff_add(x, y);
  }
  return x;
}

template <int W = 32>
__device__ __forceinline__ void warp_arg_all(float& v, int32_t& i) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int32_t oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) {
      v = ov;
      i = oi;
    }
  }
}

// ---- CTA-wide top-F selection by rank counting ----------------------------
// Keys are (value, index) under key_beats; all indices are distinct, so the
// ranks of distinct entries are distinct.  Empty entries are (-inf, INT_MAX).

constexpr int kCandCap = 512;  // candidates one CTA ranks at once

struct KeyScratch {  // shared-memory scratch of a chunk's top-F selection
  float v[kCandCap];   // qualifying candidates, unordered
  int32_t i[kCandCap];
  int count;           // candidates pushed (may pass kCandCap)
};

}  // namespace specv
