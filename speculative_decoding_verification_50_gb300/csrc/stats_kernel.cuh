// Kernel A of the hot path: one streaming pass over every logit row.
//
// a1 row statistics ("Lecture 5 - Speculative Decoding and SpecInfer" §2.1:
// temperature T gives softmax(z/T), greedy gives the one-hot argmax) and, in
// the modes that predict outcomes, the per-chunk candidates for a4 ("Speculative
// Speculative Decoding" §4.1.1: top-F draft tokens at each lookahead, the token
// sent for verification there excluded).
//
// A unit is one (batch row b, position i), i in [0, K]; a work item is one
// chunk of the unit's rows (target row i and/or draft row i): `iters` trips of
// kVecs 16-byte vectors per row per thread of a 256-thread group.  Three ways
// to stream a chunk, all with the same vector -> thread mapping (so the same
// results):
//   - register path (any layout): one CTA per item, element-wise loads,
//     software-pipelined;
//   - staged path (16-byte aligned rows): one CTA per item; thread 0 keeps a
//     ring of 1-D bulk copies (TMA) of the next trips in flight into shared
//     memory while the CTA consumes the current one;
//   - persistent path (16-byte aligned rows): every CTA loops over items and
//     a producer warp keeps the ring filled across item boundaries.
//
// Per chunk the consumers write a ChunkRec: online (max, sum 2^((z-max) log2(e)/T))
// of each row, or its first argmax for greedy rows.  With outcome prediction
// they also write the chunk's own top-F of the draft row: the per-warp
// maxima bound the chunk's top-F from below, each thread keeps the group
// holding its maximum in registers, so only the few threads with a second
// group above the bound read their share again (from L2, just streamed; one
// round trip per warp), and the qualifying logits are ranked in parallel in
// shared memory.  A chunk of a single row streams through half-size ring
// stages (twice the trips in flight).
#pragma once

#include "specv_device.cuh"

namespace specv {

// verify: target and draft rows; ssd: plus draft row K and candidates;
// predict: draft rows 0..K, candidates, no temperature; sample: one draft row
// per batch row (K = 0) with its temperature and candidates (no exclusion);
// mss: one target and one draft row per token-tree node (K = 0).
enum : int { kModeVerify = 0, kModeSsd = 1, kModePredict = 2, kModeSample = 3, kModeMss = 4 };

// Streams target rows; keeps top-F candidates; uses the temperature.
__host__ __device__ constexpr bool mode_has_target(int m) {
  return m == kModeVerify || m == kModeSsd || m == kModeMss;
}
__host__ __device__ constexpr bool mode_has_topf(int m) {
  return m == kModeSsd || m == kModePredict || m == kModeSample;
}
__host__ __device__ constexpr bool mode_has_temp(int m) { return m != kModePredict; }
constexpr int kVecs = 2;  // 16-byte vectors per row per thread per loop trip
constexpr int kMaxStages = 8;
constexpr int kTripBytes = kVecs * kThreads * 16;  // one row's share of a trip (8 KB)

struct ChunkRec {        // 48 bytes per (unit, chunk)
  float mt, st, md, sd;  // temperature rows: max and sum of 2^((z-max)c)
  float bt, bd;          // greedy rows: best logit
  int32_t it, id;        // greedy rows: first index of the best logit
  int32_t bad;           // bit 0: NaN or +inf seen in a greedy row (T > 0: shows
                         // as a NaN sum); bit 1: a staged copy did not land in time
  int32_t pad[3];
};
static_assert(sizeof(ChunkRec) == 48, "ChunkRec layout");

// A record written by another CTA, possibly of the same launch: read through
// L2 (ld.global.cg), never from a line this SM may hold from before.
__device__ __forceinline__ ChunkRec ld_rec(const ChunkRec* p) {
  const float4* q = reinterpret_cast<const float4*>(p);
  const float4 a = __ldcg(q), b = __ldcg(q + 1), c = __ldcg(q + 2);
  ChunkRec r;
  r.mt = a.x; r.st = a.y; r.md = a.z; r.sd = a.w;
  r.bt = b.x; r.bd = b.y; r.it = __float_as_int(b.z); r.id = __float_as_int(b.w);
  r.bad = __float_as_int(c.x); r.pad[0] = __float_as_int(c.y); r.pad[1] = __float_as_int(c.z);
  r.pad[2] = __float_as_int(c.w);
  return r;
}

// A sampled row's chunk may be split in up to kMaxPieces equal pieces, whose
// draft statistics (max, sum of 2^((z-max)c)) the kernel also writes, to a
// table of kMaxPieces entries per chunk.
constexpr int kMaxPieces = 8;

struct StatsParams {
  const void* zt;
  int64_t t_bs, t_rs;
  const void* zd;
  int64_t d_bs, d_rs;
  const int32_t* tokens;
  const float* temp;
  ChunkRec* recs;     // [units * nchunk]
  float* cand_v;      // [units * nchunk * F] (predict / ssd)
  int32_t* cand_i;
  int32_t B, K, V, F, nchunk, chunk, iters;  // chunk = iters * kVecs * 256 * VW logits
  int32_t fk[kMaxK + 1];  // candidates a chunk at position k keeps (<= F; the rest of its
                          // F slots padded): the fan-out, at least the Saguaro F_s
  int32_t stages;     // ring stages of the staged paths, 2..kMaxStages
  int32_t piece;      // sampler rows: trips per recorded piece of a chunk (0: none)
  int32_t pieces;     //   and pieces per chunk (2, 4 or 8)
  float2* piece_stats;  // [units * nchunk * kMaxPieces] (max, sum) of each piece
  const int32_t* cu;  // per-row draft counts (inclusive prefix sums), or null
  int32_t ntok;       // with cu: packed draft rows the buffers hold
  int32_t stall;      // test hook: 1 + the item whose first stage waits for 16
                      // bytes no copy brings, so its wait runs out (0: none)
};

// Where batch row b's logit rows, draft tokens and uniforms live: the strided
// [B, K(+1), V] layout, or rows packed by per-row draft counts ("Speculative
// Decoding" dl-note Appendix, cu_num_draft_tokens): K_b = cu[b] - cu[b-1]
// drafts, target row i at (cu[b-1] + b + i), draft row i at cu[b-1] + i,
// tokens at cu[b-1] + i, uniforms at cu[b-1] + b + i.  Counts outside
// [0, K] or past the ntok packed rows give kb = -1: the row is read nowhere.
struct RowLayout {
  int kb;          // drafts of the row (K when strided), -1 if its counts are bad
  int64_t t_off;   // element offset of its target row 0
  int64_t d_off;   // element offset of its draft row 0
  int64_t tok0;    // index of its first draft token (and of its p/q outputs)
  int64_t u_off;   // index of its first uniform
};

__device__ __forceinline__ RowLayout row_layout(const int32_t* cu, int ntok, int b, int K,
                                                int64_t t_bs, int64_t t_rs, int64_t d_bs,
                                                int64_t d_rs) {
  RowLayout L;
  if (!cu) {
    L.kb = K;
    L.t_off = static_cast<int64_t>(b) * t_bs;
    L.d_off = static_cast<int64_t>(b) * d_bs;
    L.tok0 = static_cast<int64_t>(b) * K;
    L.u_off = static_cast<int64_t>(b) * (K + 1);
    return L;
  }
  const int64_t c0 = b > 0 ? cu[b - 1] : 0, c1 = cu[b];
  const bool ok = c0 >= 0 && c1 >= c0 && c1 - c0 <= K && c1 <= ntok;
  L.kb = ok ? static_cast<int>(c1 - c0) : -1;
  const int64_t base = ok ? c0 : 0;
  L.t_off = (base + b) * t_rs;
  L.d_off = base * d_rs;
  L.tok0 = base;
  L.u_off = base + b;
  return L;
}

// log2(e)/T for a valid temperature; greedy rows and bad temperatures use 1.
__device__ __forceinline__ float temp_scale(float T) {
  return (T > 0.f && T < pos_inf()) ? __fdiv_rn(1.44269504088896341f, T) : 1.f;
}

// ---- a thread's accumulators -------------------------------------------------
// A thread streams its share of a chunk one trip at a time: a group of N =
// kVecs*VW logits of each row (kVecs vectors; logits base[k] .. base[k]+VW-1
// in vector k, in increasing index order).  Per group the max is taken once
// (three-input max) and the sums are rescaled once, branch-free; the
// exponents are computed in paired fp32 lanes.

template <int N>
__device__ __forceinline__ float group_max(const float (&z)[N], float init) {
  float r = init;
#pragma unroll
  for (int k = 0; k + 1 < N; k += 2) r = max3(r, z[k], z[k + 1]);
  return r;
}

template <int N>
__device__ __forceinline__ float group_max_nan(const float (&z)[N]) {
  float r = z[0];
#pragma unroll
  for (int k = 1; k + 1 < N; k += 2) r = max3_nan(r, z[k], z[k + 1]);
  return (N % 2 == 0) ? max3_nan(r, z[N - 1], z[N - 1]) : r;
}

// Temperature rows: online max m and sum of 2^((z-m)c), as four partial sums
// held in two pairs.  A NaN logit makes the sum NaN; a +inf logit makes it
// NaN as well (inf - inf); a row of -inf leaves m = kNegMax and the sum 0.
template <int N>
struct SoftG {
  float m;
  uint64_t s0, s1;
  __device__ __forceinline__ void init() {
    m = kNegMax;
    s0 = s1 = f2(0.f, 0.f);
  }
  __device__ __forceinline__ void add(const float (&z)[N], float c) { add_max(z, c, group_max(z, m)); }
  // mn: max(m, the group's max), NaN ignored (taken once per group when the
  // outcome-prediction tracking needs the group's own max as well)
  __device__ __forceinline__ void add_max(const float (&z)[N], float c, float mn) {
    static_assert(N % 4 == 0, "groups of whole pairs of pairs");
    const float f = ex2(__fmul_rn(__fsub_rn(m, mn), c));  // exactly 1 when m is unchanged
    const uint64_t ff = f2(f, f);
    s0 = f2_mul(s0, ff);
    s1 = f2_mul(s1, ff);
    const uint64_t mm = f2(mn, mn), cc = f2(c, c);
#pragma unroll
    for (int k = 0; k < N; k += 4) {
      float a, b, d, e;
      f2_split(f2_mul(f2_sub(f2(z[k], z[k + 1]), mm), cc), a, b);
      f2_split(f2_mul(f2_sub(f2(z[k + 2], z[k + 3]), mm), cc), d, e);
      s0 = f2_add(s0, f2(ex2(a), ex2(b)));
      s1 = f2_add(s1, f2(ex2(d), ex2(e)));
    }
    m = mn;
  }
  __device__ __forceinline__ float total() const {
    float a, b, d, e;
    f2_split(s0, a, b);
    f2_split(s1, d, e);
    return (a + b) + (d + e);
  }
};

// Greedy rows: first argmax, and whether a NaN or +inf was seen.
template <int N>
struct ArgG {
  float best;
  int32_t idx;
  int32_t bad;
  __device__ __forceinline__ void init() {
    best = neg_inf();
    idx = INT_MAX;
    bad = 0;
  }
  template <int VW>
  __device__ __forceinline__ void add(const float (&z)[N], const int32_t (&base)[N / VW]) {
    const float vm = group_max_nan(z);  // NaN if any logit is NaN
    bad |= !(vm < pos_inf());
    if (vm > best) {  // a new best: the first logit of the group equal to it
      int32_t id = INT_MAX;
#pragma unroll
      for (int k = N - 1; k >= 0; --k)
        if (z[k] == vm) id = base[k / VW] + k % VW;
      best = vm;
      idx = id;
    }
  }
};

// Outcome prediction: the group holding this thread's largest draft logit,
// kept in registers (m1, its trip t1, its logits z), and the largest maximum
// of the thread's other groups (m2), all updated without a branch.  A thread
// whose m2 is below a bound holds every logit at or above it in z.
template <int N>
struct BestGroup {
  float m1, m2;
  int t1;
  float z[N];
  __device__ __forceinline__ void init() {
    m1 = m2 = neg_inf();
    t1 = 0;
#pragma unroll
    for (int k = 0; k < N; ++k) z[k] = neg_inf();
  }
  __device__ __forceinline__ void add(const float (&zz)[N], int t) {
    add_max(zz, t, group_max(zz, neg_inf()));  // NaN ignored
  }
  // vm: the group's max, NaN ignored
  __device__ __forceinline__ void add_max(const float (&zz)[N], int t, float vm) {
    const bool nb = vm > m1;
    m2 = nb ? m1 : fmaxf(m2, vm);
    t1 = nb ? t : t1;
    m1 = nb ? vm : m1;
#pragma unroll
    for (int k = 0; k < N; ++k) z[k] = nb ? zz[k] : z[k];
  }
};

template <int VW>
struct Acc {
  static constexpr int N = kVecs * VW;
  SoftG<N> st, sd;   // temperature rows: target, draft
  ArgG<N> at, ad;    // greedy rows: target, draft
  BestGroup<N> kd;   // draft row, outcome prediction
  __device__ __forceinline__ void init() {
    st.init();
    sd.init();
    at.init();
    ad.init();
    kd.init();
  }
  // Group of trip t of the target (DRAFT = false) or draft row.
  template <bool GREEDY, bool DRAFT, bool TOPF>
  __device__ __forceinline__ void add(const float (&z)[N], const int32_t (&base)[kVecs], float c,
                                      int t) {
    if (!GREEDY && DRAFT && TOPF) {  // one group max serves both (max is exact)
      const float gz = group_max(z, neg_inf());
      sd.add_max(z, c, fmaxf(sd.m, gz));
      kd.add_max(z, t, gz);
      return;
    }
    if (GREEDY) (DRAFT ? ad : at).template add<VW>(z, base);
    else (DRAFT ? sd : st).add(z, c);
    if (DRAFT && TOPF) kd.add(z, t);
  }
};

// Unpacks vector k of a trip into its slot of the group (or -inf when absent).
template <int DT>
__device__ __forceinline__ void put_vec(float* z, const typename Elem<DT>::Vec& w) {
  float y[Elem<DT>::VW];
  Elem<DT>::unpack(w, y);
#pragma unroll
  for (int e = 0; e < Elem<DT>::VW; ++e) z[e] = y[e];
}
template <int DT>
__device__ __forceinline__ void put_none(float* z) {
#pragma unroll
  for (int e = 0; e < Elem<DT>::VW; ++e) z[e] = neg_inf();
}

// ---- register path ------------------------------------------------------------

template <int DT, bool VEC>
__device__ __forceinline__ void load_trip(const void* row, int64_t v0, int64_t v1, int nv, int it,
                                          typename Elem<DT>::Vec (&w)[kVecs]) {
#pragma unroll
  for (int k = 0; k < kVecs; ++k) {
    const int j = (it * kVecs + k) * kThreads + threadIdx.x;
    if (j < nv) w[k] = load_vec<DT, VEC>(row, v0, v1, j);
  }
}

template <int DT, bool GREEDY, bool DRAFT, bool TOPF>
__device__ __forceinline__ void consume_trip(const typename Elem<DT>::Vec (&w)[kVecs], int nv,
                                             int it, int64_t v0, float c, Acc<Elem<DT>::VW>& A) {
  constexpr int VW = Elem<DT>::VW;
  float z[kVecs * VW];
  int32_t base[kVecs];
#pragma unroll
  for (int k = 0; k < kVecs; ++k) {
    const int j = (it * kVecs + k) * kThreads + threadIdx.x;
    base[k] = static_cast<int32_t>(v0) + j * VW;
    if (j < nv) put_vec<DT>(z + k * VW, w[k]); else put_none<DT>(z + k * VW);
  }
  A.template add<GREEDY, DRAFT, TOPF>(z, base, c, it);
}

// Streams the CTA's chunk of one or two rows (software-pipelined).
template <int DT, bool VEC, bool GREEDY, bool KT, bool TOPF>
__device__ __forceinline__ void stream_chunk(const void* rowt, const void* rowd, bool has_d,
                                             int64_t v0, int64_t v1, int nv, int iters, float c,
                                             Acc<Elem<DT>::VW>& A) {
  using Vec = typename Elem<DT>::Vec;
  Vec at0[kVecs], ad0[kVecs], at1[kVecs], ad1[kVecs];
  if (KT) load_trip<DT, VEC>(rowt, v0, v1, nv, 0, at0);
  if (has_d) load_trip<DT, VEC>(rowd, v0, v1, nv, 0, ad0);
  for (int it = 0; it < iters; it += 2) {
    if (it + 1 < iters) {
      if (KT) load_trip<DT, VEC>(rowt, v0, v1, nv, it + 1, at1);
      if (has_d) load_trip<DT, VEC>(rowd, v0, v1, nv, it + 1, ad1);
    }
    if (KT) consume_trip<DT, GREEDY, false, TOPF>(at0, nv, it, v0, c, A);
    if (has_d) consume_trip<DT, GREEDY, true, TOPF>(ad0, nv, it, v0, c, A);
    if (it + 1 < iters) {
      if (it + 2 < iters) {
        if (KT) load_trip<DT, VEC>(rowt, v0, v1, nv, it + 2, at0);
        if (has_d) load_trip<DT, VEC>(rowd, v0, v1, nv, it + 2, ad0);
      }
      if (KT) consume_trip<DT, GREEDY, false, TOPF>(at1, nv, it + 1, v0, c, A);
      if (has_d) consume_trip<DT, GREEDY, true, TOPF>(ad1, nv, it + 1, v0, c, A);
    }
  }
}

// ---- one chunk of one unit ----------------------------------------------------
// Work item `item` = (unit u = item / nchunk, chunk item % nchunk); unit u is
// (batch row b, position i) = (u / (K+1), u % (K+1)).
struct Chunk {
  int b, i;
  const char* rowt;  // target row i, or null when it is not streamed
  const char* rowd;  // draft row i, or null when there is none
  int64_t v0, v1;    // the chunk covers logits [v0, v1) of its rows
  int nv;            // 16-byte vectors covering them (the last may be partial)
};

template <int DT, int MODE>
__device__ __forceinline__ Chunk chunk_at(const StatsParams& P, int64_t item) {
  using E = Elem<DT>;
  Chunk C;
  const int64_t u = item / P.nchunk;
  const int ch = static_cast<int>(item % P.nchunk);
  C.b = static_cast<int>(u / (P.K + 1));
  C.i = static_cast<int>(u % (P.K + 1));
  const RowLayout L = row_layout(P.cu, P.ntok, C.b, P.K, P.t_bs, P.t_rs, P.d_bs, P.d_rs);
  const bool live = C.i <= L.kb;  // positions past the row's drafts hold no rows
  // Verification reads draft rows i < K_b (none without draft logits);
  // prediction reads draft rows 0..K.
  const bool has_d = live && ((MODE == kModeVerify) ? (C.i < L.kb && P.zd != nullptr) : true);
  C.rowt = (mode_has_target(MODE) && live)
               ? static_cast<const char*>(P.zt) + (L.t_off + static_cast<int64_t>(C.i) * P.t_rs) * E::ES
               : nullptr;
  C.rowd = has_d ? static_cast<const char*>(P.zd) + (L.d_off + static_cast<int64_t>(C.i) * P.d_rs) * E::ES
                 : nullptr;
  C.v0 = static_cast<int64_t>(ch) * P.chunk;
  C.v1 = live ? min(static_cast<int64_t>(P.V), C.v0 + P.chunk) : C.v0;
  C.nv = static_cast<int>((C.v1 - C.v0 + E::VW - 1) / E::VW);
  return C;
}

// The draft token sent for verification at the chunk's position, excluded
// from its outcome keys (none at position K, or without candidates).
template <int MODE>
__device__ __forceinline__ int excluded_token(const StatsParams& P, const Chunk& C) {
  return (mode_has_topf(MODE) && C.i < P.K) ? P.tokens[static_cast<int64_t>(C.b) * P.K + C.i] : -1;
}

// Shared scratch of a chunk's epilogue.
struct EpiSmem {
  ChunkRec wrec[kWarps];
  float wthr[kWarps];    // each warp's g-th largest per-thread maximum
  float wthr_f[kWarps];  // each warp's (F+1)-th largest
  float wl_v[kWarps][kMaxF];
  int32_t wl_i[kWarps][kMaxF];
  KeyScratch KS;
};

__device__ __forceinline__ void push_key(KeyScratch& KS, float v, int32_t i) {
  const int slot = atomicAdd(&KS.count, 1);
  if (slot < kCandCap) {
    KS.v[slot] = v;
    KS.i[slot] = i;
  }
}

// Epilogue of chunk `item`, run by the kThreads threads of warps 0..7 after
// they have streamed it: reduces their accumulators into the chunk's ChunkRec
// (warp, then warp 0 over the eight warp partials) and, with outcome
// prediction, writes the chunk's top-F draft candidates.  `ok` is false on a
// thread whose staged copies did not all land.  Ends with a barrier, so the
// scratch is free for the next chunk.
template <int DT, bool VEC, int MODE>
__device__ __forceinline__ void chunk_finish(const StatsParams& P, const Chunk& C, int64_t item,
                                             bool greedy, float c, Acc<Elem<DT>::VW>& A, bool ok,
                                             EpiSmem& S, int excl, float2* snap = nullptr,
                                             int npieces = 0) {
  using E = Elem<DT>;
  constexpr int VW = E::VW;
  constexpr bool kTopF = mode_has_topf(MODE);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (greedy) {
    float bt = A.at.best, bd = A.ad.best;
    int32_t it = A.at.idx, id = A.ad.idx;
    warp_arg_all(bt, it);
    warp_arg_all(bd, id);
    const int bad = __any_sync(0xffffffffu, A.at.bad | A.ad.bad);
    if (lane == 0) {
      S.wrec[warp].bt = bt; S.wrec[warp].it = it; S.wrec[warp].bd = bd; S.wrec[warp].id = id;
      S.wrec[warp].bad = bad;
    }
  } else {  // (a row the chunk does not have keeps its empty statistics)
    float mt = A.st.m, s_t = A.st.total(), md = A.sd.m, s_d = A.sd.total();
    if (C.rowt) warp_soft_all(mt, s_t, c);
    if (C.rowd) warp_soft_all(md, s_d, c);  // with pieces: the last one
    if (snap) {  // the warp's last piece joins the others; the chunk is their sum (lane k: piece k)
      if (lane == 0) snap[(npieces - 1) * kWarps + warp] = make_float2(md, s_d);
      __syncwarp();
      md = kNegMax;
      s_d = 0.f;
      if (lane < npieces) {
        const float2 h = snap[lane * kWarps + warp];
        md = h.x;
        s_d = h.y;
      }
      warp_soft_all(md, s_d, c);
    }
    if (lane == 0) {
      S.wrec[warp].mt = mt; S.wrec[warp].st = s_t; S.wrec[warp].md = md; S.wrec[warp].sd = s_d;
    }
  }
  if (kTopF) {
    if (threadIdx.x == 0) S.KS.count = 0;
    // Bound: with g = ceil((F+1)/8), every warp holds g distinct logits at or
    // above its g-th largest per-thread maximum (bitonic sort of the 32
    // maxima), so at least 8g >= F+1 distinct logits reach the smallest of
    // the eight, and at least F of them are not the excluded token: a lower
    // bound on the chunk's top-F without it.
    float s = A.kd.m1;  // this thread's draft maximum
    float tw, tf;
    const int Fu = P.fk[C.i];  // candidates this chunk keeps
    if (Fu < kWarps) {
      // g = 1: the warp's largest maximum.  A warp with no finite maximum
      // (a short chunk) leaves the bound unset and the chunk takes the exact
      // path below.
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, o));
      tw = s;
      tf = neg_inf();
    } else {
#pragma unroll
      for (int k2 = 2; k2 <= 32; k2 <<= 1) {
#pragma unroll
        for (int j2 = k2 >> 1; j2 > 0; j2 >>= 1) {
          const float o = __shfl_xor_sync(0xffffffffu, s, j2);
          const bool take_max = ((lane & k2) == 0) == ((lane & j2) == 0);
          s = take_max ? fmaxf(s, o) : fminf(s, o);
        }
      }
      tw = __shfl_sync(0xffffffffu, s, (Fu + kWarps) / kWarps - 1);
      // Fallback when some warp holds fewer than g finite maxima (a short last
      // chunk): the largest, over warps, of a warp's (F+1)-th largest maximum.
      tf = (Fu < 32) ? __shfl_sync(0xffffffffu, s, Fu) : neg_inf();
    }
    if (lane == 0) {
      S.wthr[warp] = tw;
      S.wthr_f[warp] = tf;
    }
  }
  const bool copy_bad = cons_sync_or(!ok);  // a chunk copy gave up on some thread
  if (warp == 0) {
    ChunkRec r;
    r.mt = kNegMax; r.st = 0.f; r.md = kNegMax; r.sd = 0.f;
    r.bt = neg_inf(); r.it = INT_MAX; r.bd = neg_inf(); r.id = INT_MAX; r.bad = 0;
    r.pad[0] = r.pad[1] = r.pad[2] = 0;
    if (greedy) {
      float bt = neg_inf(), bd = neg_inf();
      int32_t it = INT_MAX, id = INT_MAX;
      int bad = 0;
      if (lane < kWarps) {
        bt = S.wrec[lane].bt; it = S.wrec[lane].it; bd = S.wrec[lane].bd; id = S.wrec[lane].id;
        bad = S.wrec[lane].bad;
      }
      warp_arg_all(bt, it);
      warp_arg_all(bd, id);
      r.bt = bt; r.it = it; r.bd = bd; r.id = id;
      r.bad = __any_sync(0xffffffffu, bad);
    } else {
      float mt = kNegMax, s_t = 0.f, md = kNegMax, s_d = 0.f;
      if (lane < kWarps) {
        mt = S.wrec[lane].mt; s_t = S.wrec[lane].st; md = S.wrec[lane].md; s_d = S.wrec[lane].sd;
      }
      if (C.rowt) warp_soft_all<kWarps>(mt, s_t, c);
      if (C.rowd) warp_soft_all<kWarps>(md, s_d, c);
      r.mt = mt; r.st = s_t; r.md = md; r.sd = s_d;
    }
    if (copy_bad) r.bad |= 2;
    if (lane == 0) P.recs[item] = r;
  }
  if (snap && !greedy && warp < npieces) {  // warp k: piece k over the CTA
    float m = kNegMax, z = 0.f;
    if (lane < kWarps) {
      const float2 h = snap[warp * kWarps + lane];
      m = h.x;
      z = h.y;
    }
    warp_soft_all<kWarps>(m, z, c);
    if (lane == 0) P.piece_stats[item * kMaxPieces + warp] = make_float2(m, z);
  }

  if (kTopF) {
    // Every draft logit of the chunk at or above the bound, the excluded token
    // left out, goes into a shared buffer ranked in parallel.  Only threads
    // whose maximum reaches the bound can hold one.  If the thread's other
    // groups all stay below the bound, its qualifying logits are all in the
    // group it kept in registers and it pushes them from there; otherwise
    // (rare) its share is read again by its whole warp at once -- lane l
    // fetches vector l, l+32, ... of the list (candidate, vector k).  Too many
    // qualifiers (ties at the bound), or no finite bound at all (masked rows,
    // chunks with fewer than F+1 finite logits), take the exact warp-list path.
    const int F = P.fk[C.i];  // candidates kept; the output holds P.F slots
    float thr = S.wthr[0], thr_f = S.wthr_f[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) {
      thr = fminf(thr, S.wthr[w]);
      thr_f = fmaxf(thr_f, S.wthr_f[w]);
    }
    if (!(thr > kNegMax)) thr = thr_f;
    const bool bounded = thr > kNegMax;
    const int ntrips = P.iters * kVecs;  // vectors per thread per row
    const bool cand = bounded && A.kd.m1 >= thr;
    const bool reread = cand && A.kd.m2 >= thr;
    if (cand && !reread) {
      const int j0 = A.kd.t1 * kVecs * kThreads + threadIdx.x;
#pragma unroll
      for (int k = 0; k < kVecs * VW; ++k) {
        const int32_t vi = static_cast<int32_t>(C.v0) + (j0 + (k / VW) * kThreads) * VW + k % VW;
        if (A.kd.z[k] >= thr && vi != excl) push_key(S.KS, A.kd.z[k], vi);
      }
    }
    const unsigned cm = __ballot_sync(0xffffffffu, reread);
    const int todo = __popc(cm) * ntrips;
    for (int r0 = 0; r0 < todo; r0 += 4 * 32) {
      typename E::Vec w[4];
      int jv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int idx = r0 + q * 32 + lane;
        jv[q] = -1;
        if (idx < todo) {
          const int cand = idx / ntrips;
          const int owner = warp * 32 + static_cast<int>(__fns(cm, 0, cand + 1));
          const int j = (idx - cand * ntrips) * kThreads + owner;
          if (j < C.nv) {
            jv[q] = j;
            w[q] = load_vec<DT, VEC>(C.rowd, C.v0, C.v1, j);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (jv[q] >= 0) {
          float z[VW];
          E::unpack(w[q], z);
          const int32_t base = static_cast<int32_t>(C.v0) + jv[q] * VW;
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            const int32_t vi = base + e;
            if (vi < C.v1 && vi != excl && z[e] >= thr) push_key(S.KS, z[e], vi);
          }
        }
      }
    }
    if (!bounded && threadIdx.x == 0) S.KS.count = kCandCap + 1;  // exact path below
    cons_sync();
    const int m = S.KS.count;
    float* outv = P.cand_v + item * P.F;
    int32_t* outi = P.cand_i + item * P.F;
    if (m <= kCandCap) {
      // distinct indices: the ranks are 0..m-1, each written once; slots
      // m..F-1 (fewer candidates than F) are padded
      for (int e = threadIdx.x; e < m; e += kThreads) {
        const float v = S.KS.v[e];
        const int32_t ii = S.KS.i[e];
        int rank = 0;
        for (int o = 0; o < m; ++o) rank += key_beats(S.KS.v[o], S.KS.i[o], v, ii);
        if (rank < F) {
          outv[rank] = v;
          outi[rank] = ii;
        }
      }
      if (threadIdx.x >= min(m, F) && threadIdx.x < P.F) {
        outv[threadIdx.x] = neg_inf();
        outi[threadIdx.x] = INT_MAX;
      }
    } else {
      WarpTopF L;
      L.init();
      for (int k = 0; k < ntrips; ++k) {
        const int j = k * kThreads + threadIdx.x;
        float z[VW];
        if (j < C.nv) {
          E::unpack(load_vec<DT, VEC>(C.rowd, C.v0, C.v1, j), z);
        } else {
#pragma unroll
          for (int e = 0; e < VW; ++e) z[e] = neg_inf();
        }
        const int32_t base = static_cast<int32_t>(C.v0) + j * VW;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          const int32_t vi = base + e;
          const bool pass = j < C.nv && vi < C.v1 && vi != excl && (!bounded || z[e] >= thr) &&
                            key_beats(z[e], vi, L.tv, L.ti);
          unsigned mm = __ballot_sync(0xffffffffu, pass);
          while (mm) {
            const int src = __ffs(mm) - 1;
            mm &= mm - 1;
            const float zz = __shfl_sync(0xffffffffu, z[e], src);
            const int32_t jj = __shfl_sync(0xffffffffu, vi, src);
            L.insert(zz, jj, F, lane);
          }
        }
      }
      if (lane < F) {
        S.wl_v[warp][lane] = L.v;
        S.wl_i[warp][lane] = L.i;
      }
      cons_sync();
      if (warp == 0) {
        merge_lists(S.wl_v, S.wl_i, kWarps, F, lane, outv, outi);
        if (lane >= F && lane < P.F) {
          outv[lane] = neg_inf();
          outi[lane] = INT_MAX;
        }
      }
    }
  }
  cons_sync();
}

// ---- staged paths: bulk copies into a ring of shared-memory stages --------------
// Stage s holds one trip of each streamed row: the target's share at offset 0,
// the draft's at kTripBytes.

struct RingBars {
  uint64_t full[kMaxStages];   // completes when stage s has landed
  uint64_t empty[kMaxStages];  // persistent path: all consumer warps are done with stage s
  int abort;                   // persistent path: set once a wait has given up
};

__device__ __forceinline__ int ring_trips(int nv) {
  return (nv + kVecs * kThreads - 1) / (kVecs * kThreads);
}

// Copies trip t of chunk C into stage s, completing on `full`.  Whole 16-byte
// units only (the consumers load a ragged tail themselves); the expected byte
// count is armed even when nothing is copied, so the phase completes anyway.
// A stage holds the trip of both rows (target at +0, draft at +kTripBytes);
// with `one` (a chunk of a single row) stages are kTripBytes apart and hold
// that row alone, so the same ring carries twice as many trips.
template <int DT>
__device__ __forceinline__ void ring_issue(uint64_t* full, unsigned char* ring, int s, int t,
                                           const Chunk& C, bool one = false, bool stream = true) {
  using E = Elem<DT>;
  const int64_t off = static_cast<int64_t>(t) * kTripBytes;
  int64_t bytes = (C.v1 - C.v0) * E::ES - off;
  if (bytes > kTripBytes) bytes = kTripBytes;
  if (bytes < 0) bytes = 0;
  const uint32_t b32 = static_cast<uint32_t>(bytes) & ~15u;
  const uint32_t nrows = (C.rowt ? 1u : 0u) + (C.rowd ? 1u : 0u);
  mbar_arrive_expect_tx(full, b32 * nrows);
  if (b32) {
    const int64_t src = C.v0 * E::ES + off;
    if (one) {
      bulk_load(ring + static_cast<int64_t>(s) * kTripBytes, (C.rowt ? C.rowt : C.rowd) + src, b32, full,
                stream);
    } else {
      unsigned char* base = ring + static_cast<int64_t>(s) * 2 * kTripBytes;
      if (C.rowt) bulk_load(base, C.rowt + src, b32, full, stream);
      if (C.rowd) bulk_load(base + kTripBytes, C.rowd + src, b32, full, stream);
    }
  }
}

// Accumulates this thread's vectors of trip t, which lies wholly inside the
// copied part of the chunk: no bounds checks (the common case).
template <int DT, bool GREEDY, bool KT, bool TOPF>
__device__ __forceinline__ void consume_stage_whole(const unsigned char* base, int t, const Chunk& C,
                                                    float c, Acc<Elem<DT>::VW>& A, int doff) {
  using E = Elem<DT>;
  using Vec = typename E::Vec;
  constexpr int VW = E::VW;
  constexpr int N = kVecs * VW;
  const int j0 = t * kVecs * kThreads + threadIdx.x;
  int32_t b[kVecs];
#pragma unroll
  for (int k = 0; k < kVecs; ++k) b[k] = static_cast<int32_t>(C.v0) + (j0 + k * kThreads) * VW;
  if (KT && C.rowt) {
    float z[N];
    const Vec* src = reinterpret_cast<const Vec*>(base);
#pragma unroll
    for (int k = 0; k < kVecs; ++k) put_vec<DT>(z + k * VW, src[k * kThreads + threadIdx.x]);
    A.template add<GREEDY, false, TOPF>(z, b, c, t);
  }
  if (C.rowd) {
    float z[N];
    const Vec* src = reinterpret_cast<const Vec*>(base + doff);
#pragma unroll
    for (int k = 0; k < kVecs; ++k) put_vec<DT>(z + k * VW, src[k * kThreads + threadIdx.x]);
    A.template add<GREEDY, true, TOPF>(z, b, c, t);
  }
}

// Trips of chunk C that lie wholly inside its copied part (for every thread).
template <int DT>
__device__ __forceinline__ int whole_trips(const Chunk& C, int64_t covered) {
  return static_cast<int>(((covered - C.v0) / Elem<DT>::VW) / (kVecs * kThreads));
}

// Accumulates this thread's vectors of trip t from the stage at `base`; a
// vector past the last whole 16-byte unit of the chunk (`covered` = first
// logit not copied) is gathered from global memory instead.
template <int DT, bool GREEDY, bool KT, bool TOPF>
__device__ __forceinline__ void consume_stage(const unsigned char* base, int t, const Chunk& C,
                                              int64_t covered, float c, Acc<Elem<DT>::VW>& A,
                                              int doff) {
  using E = Elem<DT>;
  using Vec = typename E::Vec;
  constexpr int VW = E::VW;
  constexpr int N = kVecs * VW;
  const int j0 = t * kVecs * kThreads + threadIdx.x;  // this thread's first vector of the trip
  int32_t b[kVecs];
#pragma unroll
  for (int k = 0; k < kVecs; ++k) b[k] = static_cast<int32_t>(C.v0) + (j0 + k * kThreads) * VW;
  // Whole trip in shared memory: the common case, no per-vector checks.
  const bool whole = C.v0 + static_cast<int64_t>(j0 + (kVecs - 1) * kThreads + 1) * VW <= covered;
  if (KT && C.rowt) {
    float z[N];
    const Vec* src = reinterpret_cast<const Vec*>(base);
#pragma unroll
    for (int k = 0; k < kVecs; ++k) {
      const int j = j0 + k * kThreads;
      const int64_t e = C.v0 + static_cast<int64_t>(j) * VW;
      if (whole || e + VW <= covered) put_vec<DT>(z + k * VW, src[k * kThreads + threadIdx.x]);
      else if (j < C.nv) put_vec<DT>(z + k * VW, E::gather(C.rowt, e, C.v1));
      else put_none<DT>(z + k * VW);
    }
    A.template add<GREEDY, false, TOPF>(z, b, c, t);
  }
  if (C.rowd) {
    float z[N];
    const Vec* src = reinterpret_cast<const Vec*>(base + doff);
#pragma unroll
    for (int k = 0; k < kVecs; ++k) {
      const int j = j0 + k * kThreads;
      const int64_t e = C.v0 + static_cast<int64_t>(j) * VW;
      if (whole || e + VW <= covered) put_vec<DT>(z + k * VW, src[k * kThreads + threadIdx.x]);
      else if (j < C.nv) put_vec<DT>(z + k * VW, E::gather(C.rowd, e, C.v1));
      else put_none<DT>(z + k * VW);
    }
    A.template add<GREEDY, true, TOPF>(z, b, c, t);
  }
}

template <int DT>
__device__ __forceinline__ int64_t covered_end(const Chunk& C) {
  using E = Elem<DT>;
  return C.v0 + ((((C.v1 - C.v0) * E::ES) & ~static_cast<int64_t>(15)) / E::ES);
}

// Staged path, one CTA per item: thread 0 keeps up to S trips in flight and
// refills a stage after the CTA barrier that closes its consumption.  Returns
// false (on every thread) if a wait gave up; the copies then in flight get a
// bounded wait before returning.
// piece > 0: every `piece` trips, up to the chunk's last piece, the draft
// row's running statistics, reduced over the warp, move to
// snap[k * kWarps + warp] (piece k) and start again, so the chunk's pieces
// are recorded apart (a short chunk fills the first pieces; the others stay
// empty).
// stall (test hook): stage 0 also waits for 16 bytes that no copy brings.
template <int DT, bool GREEDY, bool KT, bool TOPF>
__device__ __forceinline__ bool stream_chunk_staged(RingBars& R, unsigned char* ring, int S2,
                                                    const Chunk& C, float c, Acc<Elem<DT>::VW>& A,
                                                    bool stall, int piece = 0, int npieces = 0,
                                                    float2* snap = nullptr) {
  const int ntr = ring_trips(C.nv);
  const int64_t covered = covered_end<DT>(C);
  // A chunk of a single row (a draft row alone, or a target row with no
  // draft) splits each two-row stage in two: twice the trips in flight.
  const bool one = !(C.rowt && C.rowd);
  const int S = one ? min(2 * S2, kMaxStages) : S2;
  const int64_t sb = one ? kTripBytes : 2 * kTripBytes;  // stage stride
  const int doff = one ? 0 : kTripBytes;                 // draft row within a stage
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&R.full[s], 1);
    fence_mbar_init();
    if (stall) mbar_expect_tx(&R.full[0], 16);
    for (int t = 0; t < ntr && t < S; ++t) ring_issue<DT>(&R.full[t], ring, t, t, C, one, !TOPF);
  }
  __syncthreads();
  bool ok = true;
  int s = 0;
  uint32_t ph = 0;
  const int nwhole = whole_trips<DT>(C, covered);
  // the trip that ends the next recorded piece, and that piece
  int snap_at = (!GREEDY && piece > 0 && npieces > 1) ? piece : -1;
  int snap_k = 0;
  for (int t = 0; t < ntr; ++t) {
    if (!mbar_wait_bounded(&R.full[s], ph)) ok = false;
    const unsigned char* base = ring + static_cast<int64_t>(s) * sb;
    if (t < nwhole) consume_stage_whole<DT, GREEDY, KT, TOPF>(base, t, C, c, A, doff);
    else consume_stage<DT, GREEDY, KT, TOPF>(base, t, C, covered, c, A, doff);
    if (t + 1 == snap_at) {
      float m = A.sd.m, z = A.sd.total();
      warp_soft_all(m, z, c);
      if ((threadIdx.x & 31) == 0) snap[snap_k * kWarps + (threadIdx.x >> 5)] = make_float2(m, z);
      A.sd.init();
      ++snap_k;
      snap_at = snap_k < npieces - 1 ? snap_at + piece : -1;
    }
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) {
        int s2 = s;
        uint32_t p2 = ph;
        for (int t2 = t; t2 < ntr && t2 < t + S; ++t2) {
          mbar_wait_bounded(&R.full[s2], p2);
          if (++s2 == S) {
            s2 = 0;
            p2 ^= 1u;
          }
        }
      }
      __syncthreads();
      return false;
    }
    if (threadIdx.x == 0 && t + S < ntr) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      ring_issue<DT>(&R.full[s], ring, s, t + S, C, one, !TOPF);
    }
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
  if (!GREEDY && piece > 0) {  // a short chunk: the rest is the next piece, the others empty
    const int taken = snap_k;
    for (int k = taken; k < npieces - 1; ++k) {
      float m = kNegMax, z = 0.f;
      if (k == taken) {
        m = A.sd.m;
        z = A.sd.total();
        warp_soft_all(m, z, c);
        A.sd.init();
      }
      if ((threadIdx.x & 31) == 0) snap[k * kWarps + (threadIdx.x >> 5)] = make_float2(m, z);
    }
  }
  return ok;
}

// Resident CTAs per SM: 5 (48 registers), but 4 for bf16 rows with top-F
// candidates and for bf16 rows on the register path, which would spill at 48.
template <int DT, bool VEC, int MODE>
constexpr int stats_ctas_per_sm() {
  return (DT == 0 && (mode_has_topf(MODE) || !VEC)) ? 4 : 5;
}

// Register path (VEC = false: any layout) or staged path (VEC = true: 16-byte
// aligned rows, P.stages stages of dynamic shared memory); one CTA per item.
template <int DT, bool VEC, int MODE>
__global__ void __launch_bounds__(kThreads, (stats_ctas_per_sm<DT, VEC, MODE>())) stats_kernel(const StatsParams P) {
  constexpr bool kT = mode_has_target(MODE);
  constexpr bool kTopF = mode_has_topf(MODE);
  __shared__ EpiSmem S;
  pdl_launch_dependents();  // the decision kernel may be scheduled once every CTA has started
  const Chunk C = chunk_at<DT, MODE>(P, blockIdx.x);
  const float T = mode_has_temp(MODE) ? P.temp[C.b] : 0.f;
  const bool greedy = !mode_has_temp(MODE) || T == 0.f;
  const float c = greedy ? 1.f : temp_scale(T);
  const int excl = excluded_token<MODE>(P, C);  // fetched now, used by the epilogue
  Acc<Elem<DT>::VW> A;
  A.init();
  bool ok = true;
  // the sampler's chunks may record their pieces apart (staged path)
  __shared__ float2 snap[MODE == kModeSample ? kMaxPieces * kWarps : 1];
  const bool halves = MODE == kModeSample && VEC && !greedy && P.piece > 0;
  if (VEC) {
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ RingBars R;
    const bool stall = P.stall == static_cast<int64_t>(blockIdx.x) + 1;
    ok = greedy ? stream_chunk_staged<DT, true, kT, kTopF>(R, ring, P.stages, C, c, A, stall)
                : stream_chunk_staged<DT, false, kT, kTopF>(R, ring, P.stages, C, c, A, stall,
                                                            halves ? P.piece : 0, P.pieces, snap);
  } else if (greedy) {
    stream_chunk<DT, false, true, kT, kTopF>(C.rowt, C.rowd, C.rowd != nullptr, C.v0, C.v1, C.nv,
                                             P.iters, c, A);
  } else {
    stream_chunk<DT, false, false, kT, kTopF>(C.rowt, C.rowd, C.rowd != nullptr, C.v0, C.v1, C.nv,
                                              P.iters, c, A);
  }
  chunk_finish<DT, VEC, MODE>(P, C, blockIdx.x, greedy, c, A, ok, S, excl, halves ? snap : nullptr,
                              P.pieces);
}

// ---- persistent path ------------------------------------------------------------
// kThreads consumer threads (warps 0-7) plus one producer warp (warp 8).  A CTA
// takes the items blockIdx.x, blockIdx.x + gridDim.x, ... in order.  Lane 0 of
// the producer warp walks the same sequence of trips and copies the g-th into
// stage g mod S, once all eight consumer warps have arrived on that stage's
// empty barrier; the consumers run a chunk's epilogue while the copies of the
// next chunk are already in flight.  Every wait is bounded: after a timeout
// the CTA issues no more copies, flags every chunk it still owns (ChunkRec.bad
// bit 1) and still writes all their records.
constexpr int kRingThreads = kThreads + 32;

template <int DT, int MODE>
__device__ __forceinline__ void ring_produce(const StatsParams& P, RingBars& R, unsigned char* ring,
                                             int64_t items) {
  const int S = P.stages;
  volatile int* abort = &R.abort;
  int64_t g = 0;  // trips issued so far; the next goes to stage s with parity ph
  int s = 0;
  uint32_t ph = 0;
  for (int64_t item = blockIdx.x; item < items && !*abort; item += gridDim.x) {
    const Chunk C = chunk_at<DT, MODE>(P, item);
    const int ntr = ring_trips(C.nv);
    for (int t = 0; t < ntr; ++t) {
      if (*abort || !mbar_wait_bounded(&R.empty[s], ph ^ 1u)) {
        *abort = 1;
        break;
      }
      ring_issue<DT>(&R.full[s], ring, s, t, C);
      ++g;
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
  if (*abort) {
    // The copies that may still be in flight (the last S trips issued) get a
    // bounded wait to land before the CTA can exit.
    for (int64_t g2 = g > S ? g - S : 0; g2 < g; ++g2)
      mbar_wait_bounded(&R.full[g2 % S], static_cast<uint32_t>((g2 / S) & 1));
  }
}

// Consumes the trips of one chunk; returns false if any of them was not waited
// for successfully (its data are then garbage and the chunk is flagged).
template <int DT, bool GREEDY, bool KT, bool TOPF>
__device__ __forceinline__ bool ring_consume(RingBars& R, const unsigned char* ring, int S, int& s,
                                             uint32_t& ph, const Chunk& C, float c,
                                             Acc<Elem<DT>::VW>& A) {
  volatile int* abort = &R.abort;
  const int ntr = ring_trips(C.nv);
  const int64_t covered = covered_end<DT>(C);
  const int nwhole = whole_trips<DT>(C, covered);
  bool ok = true;
  for (int t = 0; t < ntr; ++t) {
    if (*abort) {
      ok = false;
    } else if (!mbar_wait_bounded(&R.full[s], ph)) {
      ok = false;
      *abort = 1;
    }
    const unsigned char* base = ring + static_cast<int64_t>(s) * 2 * kTripBytes;
    if (t < nwhole) consume_stage_whole<DT, GREEDY, KT, TOPF>(base, t, C, c, A, kTripBytes);
    else consume_stage<DT, GREEDY, KT, TOPF>(base, t, C, covered, c, A, kTripBytes);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&R.empty[s]);
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
  return ok;
}

template <int DT, int MODE>
__global__ void __launch_bounds__(kRingThreads, 2) stats_ring_kernel(const StatsParams P) {
  constexpr bool kT = mode_has_target(MODE);
  constexpr bool kTopF = mode_has_topf(MODE);
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ RingBars R;
  __shared__ EpiSmem S;
  const int64_t items = static_cast<int64_t>(P.B) * (P.K + 1) * P.nchunk;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&R.full[s], 1);
      mbar_init(&R.empty[s], kWarps);
    }
    R.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x >= kThreads) {
    if (threadIdx.x == kThreads) ring_produce<DT, MODE>(P, R, ring, items);
    return;
  }
  int s = 0;  // stage and parity of the next trip to consume
  uint32_t ph = 0;
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const Chunk C = chunk_at<DT, MODE>(P, item);
    const float T = mode_has_temp(MODE) ? P.temp[C.b] : 0.f;
    const bool greedy = !mode_has_temp(MODE) || T == 0.f;
    const float c = greedy ? 1.f : temp_scale(T);
    Acc<Elem<DT>::VW> A;
    A.init();
    const bool ok = greedy ? ring_consume<DT, true, kT, kTopF>(R, ring, P.stages, s, ph, C, c, A)
                           : ring_consume<DT, false, kT, kTopF>(R, ring, P.stages, s, ph, C, c, A);
    chunk_finish<DT, true, MODE>(P, C, item, greedy, c, A, ok, S, excluded_token<MODE>(P, C));
  }
}

}  // namespace specv
