// Host-side encoding of the TMA tensor maps used by the sequential kernels.
//
// The encoder (cuTensorMapEncodeTiled) is a driver entry point; it is looked
// up once through the runtime, so the library links against the CUDA runtime
// only.  A map is a 128-byte descriptor of a 3-D view of a per-token tensor:
// (channel, head, token) with the channel dimension contiguous.
#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder(cudaError_t *err) {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (status == cudaSuccess && (q != cudaDriverEntryPointSuccess || p == nullptr)) status = cudaErrorSymbolNotFound;
    if (status == cudaSuccess) fn = (EncodeTiledFn)p;
  });
  *err = status;
  return fn;
}

// [tokens][heads][dim] elements of `bytes` each (dim = 64 or 128); box = box_c
// channels x 1 head x 64 tokens.  Channels past dim (a 64-wide head) arrive as
// zeros, so the kernels' 128-wide tiles hold a zero-padded head.
cudaError_t encode(CUtensorMap *m, const void *base, int bytes, int heads, int64_t tokens, int dim, int box_c,
                   bool swz) {
  cudaError_t e;
  EncodeTiledFn fn = encoder(&e);
  if (fn == nullptr) return e;
  const cuuint64_t dims[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)(tokens > 0 ? tokens : 1)};
  const cuuint64_t strides[2] = {(cuuint64_t)dim * bytes, (cuuint64_t)dim * bytes * heads};  // bytes, dims 1 and 2
  const cuuint32_t box[3] = {(cuuint32_t)box_c, 1, (cuuint32_t)kChunk};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                        const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t make_tma_maps(const Problem &P, const void *v, const void *d, TmaMaps *out) {
  cudaError_t e;
  if ((e = encode(&out->k, P.k, 2, P.H, P.Ttot, P.K, 64, true)) != cudaSuccess) return e;
  if ((e = encode(&out->q, P.q, 2, P.H, P.Ttot, P.K, 64, true)) != cudaSuccess) return e;
  if (v != nullptr && (e = encode(&out->v, v, 2, P.HV, P.Ttot, P.V, 64, true)) != cudaSuccess) return e;
  if (d != nullptr && (e = encode(&out->d, d, 2, P.HV, P.Ttot, P.V, 64, true)) != cudaSuccess) return e;
  if (P.scalar_gate) return cudaSuccess;  // [tokens][HV] scalars: no tiled view (the kernels broadcast them)
  return encode(&out->g, P.g, 4, P.HV, P.Ttot, P.K, 128, false);
}

}  // namespace kda
