// Device helpers shared by the spec-tree kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bastion.h"

#define BST_DEV __device__ __forceinline__

namespace bst {

constexpr unsigned FULL = 0xffffffffu;

// ---------------------------------------------------------------- element types
// Element loads: f32 and bf16 logits / activations.  bf16 is kept as raw bits
// and widened exactly (bits << 16).
BST_DEV float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
BST_DEV float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xffff0000u); }

struct F32Tag {
  using storage = float;
  static constexpr int kVec = 4;  // elements per 16-byte vector
};
struct BF16Tag {
  using storage = uint16_t;
  static constexpr int kVec = 8;
};

// Unpack one 16-byte vector into kVec floats.
template <class Tag>
BST_DEV void unpack16(const uint4 &v, float *out);
template <>
BST_DEV void unpack16<F32Tag>(const uint4 &v, float *out) {
  out[0] = __uint_as_float(v.x);
  out[1] = __uint_as_float(v.y);
  out[2] = __uint_as_float(v.z);
  out[3] = __uint_as_float(v.w);
}
template <>
BST_DEV void unpack16<BF16Tag>(const uint4 &v, float *out) {
  out[0] = bf16_lo(v.x);
  out[1] = bf16_hi(v.x);
  out[2] = bf16_lo(v.y);
  out[3] = bf16_hi(v.y);
  out[4] = bf16_lo(v.z);
  out[5] = bf16_hi(v.z);
  out[6] = bf16_lo(v.w);
  out[7] = bf16_hi(v.w);
}

// Element j (0 <= j < kVec, a compile-time constant after unrolling) of a
// packed 16-byte vector.
template <class Tag>
BST_DEV float elem16(const uint4 &v, int j);
template <>
BST_DEV float elem16<F32Tag>(const uint4 &v, int j) {
  const uint32_t w = (j == 0) ? v.x : (j == 1) ? v.y : (j == 2) ? v.z : v.w;
  return __uint_as_float(w);
}
template <>
BST_DEV float elem16<BF16Tag>(const uint4 &v, int j) {
  const int q = j >> 1;
  const uint32_t w = (q == 0) ? v.x : (q == 1) ? v.y : (q == 2) ? v.z : v.w;
  return (j & 1) ? bf16_hi(w) : bf16_lo(w);
}
// Pack kVec floats of a scalar-loaded tail back into the vector form.
template <class Tag>
BST_DEV uint4 pack16(const float *f);
template <>
BST_DEV uint4 pack16<F32Tag>(const float *f) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}
template <>
BST_DEV uint4 pack16<BF16Tag>(const float *f) {
  // values came from bf16, so the upper 16 bits carry them exactly
  auto h = [](float a) { return __float_as_uint(a) >> 16; };
  return make_uint4(h(f[0]) | (h(f[1]) << 16), h(f[2]) | (h(f[3]) << 16), h(f[4]) | (h(f[5]) << 16),
                    h(f[6]) | (h(f[7]) << 16));
}

// Maximum of the kVec elements of a packed 16-byte vector.  bf16 pairs are
// compared packed (max of bf16 values is exact), then widened once.
template <class Tag>
BST_DEV float vmax16(const uint4 &v);
template <>
BST_DEV float vmax16<F32Tag>(const uint4 &v) {
  return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)), fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}
template <>
BST_DEV float vmax16<BF16Tag>(const uint4 &v) {
  uint32_t a, b2;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(b2) : "r"(v.z), "r"(v.w));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(a), "r"(b2));
  return fmaxf(bf16_lo(a), bf16_hi(a));
}

template <class Tag>
BST_DEV float load_scalar(const void *base, int64_t idx);
template <>
BST_DEV float load_scalar<F32Tag>(const void *base, int64_t idx) {
  return __ldg(reinterpret_cast<const float *>(base) + idx);
}
template <>
BST_DEV float load_scalar<BF16Tag>(const void *base, int64_t idx) {
  uint16_t b = __ldg(reinterpret_cast<const unsigned short *>(base) + idx);
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Element `idx` of a row staged in shared memory, as float (exact).
template <class Tag>
BST_DEV float load_scalar_shared(const uint8_t *stage, int idx);
template <>
BST_DEV float load_scalar_shared<F32Tag>(const uint8_t *stage, int idx) {
  return reinterpret_cast<const float *>(stage)[idx];
}
template <>
BST_DEV float load_scalar_shared<BF16Tag>(const uint8_t *stage, int idx) {
  return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(stage)[idx]) << 16);
}

// Streaming 16-byte load that does not allocate in L1 (read-once data).
BST_DEV uint4 ld_stream16(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---------------------------------------------------------------- ordering keys
// Order-preserving map float -> uint32 (larger float -> larger uint).  Finite
// floats never map to 0, which therefore marks "empty".  -0.0 and +0.0 compare
// equal as floats, so they map to the same key (that of +0.0): an ordering by
// (value, index) then breaks a tie between the two zeros by index, as a
// comparison of the float values does.
BST_DEV uint32_t sortable(float f) {
  uint32_t u = __float_as_uint(f);
  u = (u == 0x80000000u) ? 0u : u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
BST_DEV float unsortable(uint32_t s) {
  uint32_t u = (s & 0x80000000u) ? (s & 0x7fffffffu) : ~s;
  return __uint_as_float(u);
}

// (value, index) candidate ordered by value descending then index ascending.
struct Cand {
  float v;
  int32_t i;
};
BST_DEV bool better(float va, int32_t ia, float vb, int32_t ib) {
  return va > vb || (va == vb && ia < ib);
}

// 64-bit key: larger is better (value desc, index asc).
BST_DEV uint64_t pack_vi(float v, int32_t i) {
  return (static_cast<uint64_t>(sortable(v)) << 32) | static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(i));
}
BST_DEV float packed_v(uint64_t k) { return unsortable(static_cast<uint32_t>(k >> 32)); }
BST_DEV int32_t packed_i(uint64_t k) { return static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(k)); }

BST_DEV uint64_t warp_max_u64(uint64_t x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    uint64_t y = __shfl_xor_sync(FULL, x, o);
    x = y > x ? y : x;
  }
  return x;
}
BST_DEV float warp_max_f(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(FULL, x, o));
  return x;
}
BST_DEV float warp_sum_f(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(FULL, x, o);
  return x;
}

// Fetch-and-add with acquire-release semantics at GPU scope: the caller's
// earlier writes (and reductions) are visible to whoever observes the new
// value, and the caller then sees everything published before the old one.
BST_DEV uint32_t atomic_add_acq_rel_gpu(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

BST_DEV void set_err(uint32_t *err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

constexpr float kLog2e = 1.4426950408889634f;

// Programmatic dependent launch.  The four stages run back to back on one
// stream and each is launched with programmatic stream serialization, so the
// next grid may be scheduled while this one still runs.  pdl_wait() blocks
// until every grid this one depends on has completed and its writes are
// visible: a kernel calls it before its first global read or write of data a
// predecessor may touch, and does only private set-up (shared memory,
// barriers, descriptor prefetch) before it.  pdl_trigger() lets the next grid
// start launching; it does not publish anything, so it may come early.
// Without the launch attribute both are no-ops.
BST_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
BST_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Host side: the launch attributes every stage uses (programmatic
// serialization, plus a cluster shape when cluster_x > 0).  `attrs` must have
// room for two entries; returns how many were filled.
inline unsigned fill_launch_attrs(cudaLaunchAttribute *attrs, int cluster_x = 0, int cluster_y = 1) {
  unsigned n = 0;
  attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 0) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = cluster_x;
    attrs[n].val.clusterDim.y = cluster_y;
    attrs[n].val.clusterDim.z = 1;
    ++n;
  }
  return n;
}

// Host side: every kernel prefers the largest shared-memory carveout, so
// consecutive stages never need the SM's L1/shared split to be reconfigured.
template <class F>
inline cudaError_t prefer_max_shared(F *fn) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                              static_cast<int>(cudaSharedmemCarveoutMaxShared));
}

BST_DEV uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Optional phase trace (compiled in with -DBST_TRACE only): a kernel defines a
// __device__ buffer of 16 stamps per CTA and records %globaltimer at its phase
// boundaries.  Normal builds contain none of it.
#ifdef BST_TRACE
#define BST_STAMP(buf, ev)                                                                              \
  do {                                                                                                  \
    const unsigned cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);               \
    if (cta_ < 4096u && (ev) < 16) (buf)[cta_ * 16u + (ev)] = ::bst::now_ns();                          \
  } while (0)
#else
#define BST_STAMP(buf, ev) \
  do {                     \
  } while (0)
#endif

}  // namespace bst
