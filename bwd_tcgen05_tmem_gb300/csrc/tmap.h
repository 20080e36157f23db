// tmap.h -- host-side TMA tensor-map construction for [batch, token, head, d]
// views of 16-bit tensors given by element strides.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace attn {

// Position of the (head, token, batch) coordinates inside a 4-D tensor map
// whose outer dimensions are sorted by stride.  The kernel rebuilds the
// coordinate vector with `coords()`.
struct MapOrder {
  uint8_t pos_head, pos_tok, pos_batch;  // each in {1, 2, 3}
};

__host__ __device__ inline void map_coords(MapOrder o, int d, int h, int t, int b, int& c1,
                                           int& c2, int& c3) {
  c1 = (o.pos_head == 1) ? h : (o.pos_tok == 1) ? t : b;
  c2 = (o.pos_head == 2) ? h : (o.pos_tok == 2) ? t : b;
  c3 = (o.pos_head == 3) ? h : (o.pos_tok == 3) ? t : b;
  (void)d;
}

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

inline EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Build a tensor map over a 16-bit tensor with logical shape
// [batch][tokens][heads][d] (element strides s_batch, s_tok, s_head; d is
// contiguous) whose box is 64 elements of d x `box_rows` tokens, 128-byte
// swizzle, zero fill outside the tensor.  Returns 0 on success.
inline int make_row_map(CUtensorMap* map, MapOrder* order, const void* base, bool bf16, int d,
                        int heads, int64_t tokens, int batch, int64_t s_head, int64_t s_tok,
                        int64_t s_batch, int box_rows) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return -1;
  struct Dim {
    uint64_t extent;
    uint64_t stride_bytes;
    uint32_t box;
    int which;  // 0 head, 1 token, 2 batch
  } dims[3] = {{(uint64_t)heads, (uint64_t)s_head * 2, 1u, 0},
               {(uint64_t)tokens, (uint64_t)s_tok * 2, (uint32_t)box_rows, 1},
               {(uint64_t)batch, (uint64_t)s_batch * 2, 1u, 2}};
  // sort outer dims by stride (stable, 3 elements)
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j + 1 < 3 - i; ++j)
      if (dims[j].stride_bytes > dims[j + 1].stride_bytes) {
        Dim t = dims[j];
        dims[j] = dims[j + 1];
        dims[j + 1] = t;
      }
  cuuint64_t gdim[4] = {(cuuint64_t)d, dims[0].extent, dims[1].extent, dims[2].extent};
  cuuint64_t gstride[3] = {dims[0].stride_bytes, dims[1].stride_bytes, dims[2].stride_bytes};
  cuuint32_t box[4] = {64u, dims[0].box, dims[1].box, dims[2].box};
  cuuint32_t estride[4] = {1u, 1u, 1u, 1u};
  for (int i = 0; i < 3; ++i) {
    if (gdim[i + 1] == 0) return -2;
    // a size-1 dimension may carry any stride; give it a legal one
    if (gstride[i] == 0 || (gstride[i] % 16) != 0) {
      if (gdim[i + 1] == 1)
        gstride[i] = 16;
      else
        return -3;
    }
  }
  for (int i = 0; i < 3; ++i) {
    if (dims[i].which == 0) order->pos_head = (uint8_t)(i + 1);
    if (dims[i].which == 1) order->pos_tok = (uint8_t)(i + 1);
    if (dims[i].which == 2) order->pos_batch = (uint8_t)(i + 1);
  }
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   4, const_cast<void*>(base), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -4;
}

}  // namespace attn
