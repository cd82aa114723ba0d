// xp_tma.cuh -- host-side creation of TMA tensor maps (cuTensorMapEncodeTiled
// reached through the runtime's driver entry point, so the library does not
// link libcuda directly).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace xp {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor [outer, inner] with row pitch `ld` elements; box
// [box_outer, box_inner] with 128-byte swizzle (box_inner * 2 must be 128).
// Out-of-range elements of a box are filled with zeros, or with NaN when
// nan_fill is set.
inline bool make_map_bf16_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
                             uint32_t box_inner, uint32_t box_outer, bool nan_fill = false) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   nan_fill ? CU_TENSOR_MAP_FLOAT_OOB_FILL_NAN_REQUEST_ZERO_FMA : CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D tensor [outer, inner] of 2- or 4-byte elements (bf16 or fp32), row
// pitch `ld` elements, box [box_outer, box_inner] without swizzle (the box
// lands in shared memory as dense rows of box_inner elements; box_inner *
// elem_bytes must be a multiple of 16), or with the 128-byte swizzle
// (box_inner * elem_bytes == 128).  Out-of-range elements read as zero.
inline bool make_map_plain_2d(CUtensorMap* map, const void* ptr, uint32_t elem_bytes, uint64_t inner, uint64_t outer,
                              uint64_t ld, uint32_t box_inner, uint32_t box_outer, bool swizzle128 = false) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// make_map_bf16_2d through a small per-thread cache keyed on every argument,
// so repeated calls on the same buffers skip the encode.
inline bool cached_map_bf16_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
                               uint32_t box_inner, uint32_t box_outer, bool nan_fill = false) {
  struct Entry {
    const void* ptr;
    uint64_t inner, outer, ld;
    uint32_t bi, bo;
    bool nan;
    CUtensorMap map;
  };
  static thread_local Entry cache[32];
  static thread_local unsigned next = 0;
  for (auto& e : cache)
    if (e.ptr == ptr && e.inner == inner && e.outer == outer && e.ld == ld && e.bi == box_inner &&
        e.bo == box_outer && e.nan == nan_fill) {
      *map = e.map;
      return true;
    }
  if (!make_map_bf16_2d(map, ptr, inner, outer, ld, box_inner, box_outer, nan_fill)) return false;
  Entry& e = cache[next++ % 32];
  e.ptr = ptr;
  e.nan = nan_fill;
  e.inner = inner;
  e.outer = outer;
  e.ld = ld;
  e.bi = box_inner;
  e.bo = box_outer;
  e.map = *map;
  return true;
}

// make_map_plain_2d through its own small per-thread cache.
inline bool cached_map_plain_2d(CUtensorMap* map, const void* ptr, uint32_t elem_bytes, uint64_t inner,
                                uint64_t outer, uint64_t ld, uint32_t box_inner, uint32_t box_outer,
                                bool swizzle128 = false) {
  struct Entry {
    const void* ptr;
    uint64_t inner, outer, ld;
    uint32_t eb, bi, bo;
    bool sw;
    CUtensorMap map;
  };
  static thread_local Entry cache[32];
  static thread_local unsigned next = 0;
  for (auto& e : cache)
    if (e.ptr == ptr && e.eb == elem_bytes && e.inner == inner && e.outer == outer && e.ld == ld &&
        e.bi == box_inner && e.bo == box_outer && e.sw == swizzle128) {
      *map = e.map;
      return true;
    }
  if (!make_map_plain_2d(map, ptr, elem_bytes, inner, outer, ld, box_inner, box_outer, swizzle128)) return false;
  Entry& e = cache[next++ % 32];
  e.ptr = ptr;
  e.sw = swizzle128;
  e.eb = elem_bytes;
  e.inner = inner;
  e.outer = outer;
  e.ld = ld;
  e.bi = box_inner;
  e.bo = box_outer;
  e.map = *map;
  return true;
}

}  // namespace xp
