// Device helpers shared by the verification and outcome-prediction kernels.
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Row-status bits (meaning fixed by the C ABI header).
enum : int32_t {
  kBadToken = 1,
  kNonFinite = 2,
  kBadTemp = 4,
  kFallback = 8,
  kTimeout = 16,  // a staged bulk copy did not land within the wait bound
  kBadCount = 32, // per-row draft counts outside [0, K] or past the packed rows
  kErrors = kBadToken | kNonFinite | kBadTemp | kTimeout | kBadCount
};

constexpr float kNegMax = -3.402823466e+38f;  // lowest finite float

__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000); }
__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// 2^x on the SFU (PTX ex2.approx.ftz.f32): 2^-inf = 0, NaN propagates.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Paired fp32 arithmetic (two lanes of one 64-bit register, round to nearest,
// no fused multiply-add) and three-input max, native on sm_100 and later.
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three, NaN inputs ignored (NaN only if all three are NaN)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// max of three, NaN if any input is NaN
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Element traits: DT 0 = bf16 (raw 16-bit patterns), 1 = fp32.  A "vector"
// is 16 bytes: 8 bf16 or 4 fp32 logits.
template <int DT>
struct Elem;

template <>
struct Elem<0> {
  static constexpr int VW = 8;
  static constexpr int ES = 2;
  using Vec = uint4;
  using Raw = unsigned short;
  __device__ static Raw raw(const void* row, int64_t v) {
    return __ldg(reinterpret_cast<const unsigned short*>(row) + v);
  }
  __device__ static Raw neg_inf_raw() { return 0xff80u; }
  __device__ static float scalar(const void* row, int64_t v) {
    unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(row) + v);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  __device__ static Vec vec(const void* row, int64_t v) {  // v multiple of 8
    return __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(row) + v * ES));
  }
  __device__ static void unpack(const Vec& w, float (&z)[VW]) {
    z[0] = __uint_as_float(w.x << 16);
    z[1] = __uint_as_float(w.x & 0xffff0000u);
    z[2] = __uint_as_float(w.y << 16);
    z[3] = __uint_as_float(w.y & 0xffff0000u);
    z[4] = __uint_as_float(w.z << 16);
    z[5] = __uint_as_float(w.z & 0xffff0000u);
    z[6] = __uint_as_float(w.w << 16);
    z[7] = __uint_as_float(w.w & 0xffff0000u);
  }
  // Vector with elements [v, v+VW) clipped to [.., vend); missing -> -inf.
  __device__ static Vec gather(const void* row, int64_t v, int64_t vend) {
    uint32_t h[VW];
#pragma unroll
    for (int k = 0; k < VW; ++k) {
      h[k] = (v + k < vend)
                 ? static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row) + v + k))
                 : 0xff80u;
    }
    Vec w;
    w.x = h[0] | (h[1] << 16);
    w.y = h[2] | (h[3] << 16);
    w.z = h[4] | (h[5] << 16);
    w.w = h[6] | (h[7] << 16);
    return w;
  }
};

template <>
struct Elem<1> {
  static constexpr int VW = 4;
  static constexpr int ES = 4;
  using Vec = float4;
  using Raw = float;
  __device__ static Raw raw(const void* row, int64_t v) {
    return __ldg(reinterpret_cast<const float*>(row) + v);
  }
  __device__ static Raw neg_inf_raw() { return neg_inf(); }
  __device__ static float scalar(const void* row, int64_t v) {
    return __ldg(reinterpret_cast<const float*>(row) + v);
  }
  __device__ static Vec vec(const void* row, int64_t v) {
    return __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const char*>(row) + v * ES));
  }
  __device__ static void unpack(const Vec& w, float (&z)[VW]) {
    z[0] = w.x;
    z[1] = w.y;
    z[2] = w.z;
    z[3] = w.w;
  }
  __device__ static Vec gather(const void* row, int64_t v, int64_t vend) {
    float z[VW];
#pragma unroll
    for (int k = 0; k < VW; ++k)
      z[k] = (v + k < vend) ? __ldg(reinterpret_cast<const float*>(row) + v + k) : neg_inf();
    return make_float4(z[0], z[1], z[2], z[3]);
  }
};

// Load vector j of the slice [v0, v1) of `row`: elements v0 + j*VW .. +VW-1,
// -inf beyond v1.  VEC: the row base and v0 are 16-byte aligned.
template <int DT, bool VEC>
__device__ __forceinline__ typename Elem<DT>::Vec load_vec(const void* row, int64_t v0,
                                                           int64_t v1, int j) {
  using E = Elem<DT>;
  const int64_t v = v0 + static_cast<int64_t>(j) * E::VW;
  if (VEC && v + E::VW <= v1) return E::vec(row, v);
  return E::gather(row, v, v1);
}

// ---- shared-memory addresses, mbarriers, 1-D bulk (TMA) copies, cluster barrier

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Raises the byte count the barrier's current phase waits for, without an
// arrival (the test hook that makes a bounded wait run out uses it).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned) from
// global memory into this CTA's shared memory, completing on `bar`.  Logits
// read once per pass are marked evict-first (`stream`): under the stream's
// pressure the L2 then gives up those lines before the others (the kernels'
// code, the chunk records, the inputs of the decision).  A chunk whose
// epilogue reads some of its logits again (the top-F candidates) keeps the
// default policy.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          bool stream = true) {
  if (stream) {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
        "%2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
  }
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, letting the hardware suspend the thread for up to about
// `ns` nanoseconds while the phase is incomplete (woken early when it completes).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar`, giving up after about a second of device
// time (or 2^20 suspended polls): returns false on timeout instead of waiting
// forever.  The common case -- the phase already complete -- costs one poll;
// otherwise the thread sleeps in the hardware wait rather than spinning.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 0; it < (1u << 20); ++it) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (clock64() - t0 > 2000000000LL) break;
  }
  return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Named barrier 1 over the kThreads threads of warps 0..kWarps-1 (a CTA's
// whole block, or its consumer warps when a producer warp runs beside them).
__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// As cons_sync, returning whether `p` held on any of those threads.
__device__ __forceinline__ bool cons_sync_or(bool p) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n bar.red.or.pred b, 1, 256, a;\n selp.u32 %0, 1, 0, b;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(p))
      : "memory");
  return r != 0;
}

// Programmatic dependent launch: a kernel lets the next kernel on its stream
// (launched with programmatic stream serialization) start early, and that
// kernel waits for this one's completion -- memory included -- before it
// touches this one's outputs.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Split cluster barrier: arrive (release) now, wait (acquire) later.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(0xffffffffu, x, o);
  return x;  // lane 0 holds the sum
}

}  // namespace specv
