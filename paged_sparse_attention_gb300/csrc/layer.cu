// The layer step around the attention path: Q/K/V projections, the rotary position
// embedding, and the gradient ends of both.
//
// "Out of the Memory Barrier" (gist.science explainer, 2.A "Chunk-Recurrent Training
// with Activation Recomputation"): the sequence is processed chunk by chunk; the
// reverse sweep recomputes the chunk's activations (here the queries, from the layer
// input) just before its backward, and the chunk's K/V gradients, complete once every
// later chunk has run its backward, go back through the rotary embedding and the
// projections.  The models of the explainer's experiments (Qwen2.5) use the rotate-half
// rotary embedding: the pair (x[j], x[j + d/2]) of a head turned by the angle
// position * theta^(-2j/d).
//
//   oomb_gemm        plain GEMMs (projections and their gradients) on cuBLASLt, with
//                    the caller's workspace
//   bias_rope        optional bias, the rotation (forward or inverse) and the cast of a
//                    token-major [n, H, d] tensor; cos/sin of each (position, pair) are
//                    computed once per token in double precision (positions reach 4M,
//                    where a float angle keeps no fractional bits) and shared by the
//                    H heads
//   grad_gather      dK, dV of a token range from the paged gradient pool, token-major
#include <cublasLt.h>

#include <cmath>
#include <mutex>

#include "oomb_internal.h"

namespace oomb {
namespace {

constexpr int kRopeThreads = 128;
constexpr int kMaxHalf = 64;  // head_dim <= 128

template <typename T>
__device__ __forceinline__ float load_f(const T* p, size_t i);
template <>
__device__ __forceinline__ float load_f<float>(const float* p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ void store_f(T* p, size_t i, float v);
template <>
__device__ __forceinline__ void store_f<float>(float* p, size_t i, float v) { p[i] = v; }
template <>
__device__ __forceinline__ void store_f<__nv_bfloat16>(__nv_bfloat16* p, size_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

// One block per token row i: out[i, h, :] = rot_i(in[i, h, :] + bias[h, :]).
// mode 0: no rotation; 1: rotate by +angle; 2: rotate by -angle (the transpose).
template <typename TI, typename TO>
__global__ void __launch_bounds__(kRopeThreads)
    bias_rope(const TI* __restrict__ in, const float* __restrict__ bias, TO* __restrict__ out, int H, int d,
              int64_t pos0, double log2_theta, int mode) {
  __shared__ float cs[kMaxHalf], sn[kMaxHalf];
  const int i = blockIdx.x, half = d / 2;
  if (mode != 0) {
    for (int j = threadIdx.x; j < half; j += kRopeThreads) {
      const double freq = exp2(-2.0 * (double)j / (double)d * log2_theta);  // theta^(-2j/d)
      const double ang = (double)(pos0 + i) * freq;
      double s, c;
      sincos(ang, &s, &c);
      cs[j] = (float)c;
      sn[j] = mode == 2 ? -(float)s : (float)s;
    }
    __syncthreads();
  }
  const size_t row = (size_t)i * H * d;
  for (int idx = threadIdx.x; idx < H * half; idx += kRopeThreads) {
    const int h = idx / half, j = idx % half;
    const size_t ia = row + (size_t)h * d + j, ib = ia + half;
    float a = load_f<TI>(in, ia), b = load_f<TI>(in, ib);
    if (bias) {
      a += bias[h * d + j];
      b += bias[h * d + j + half];
    }
    if (mode != 0) {
      const float c = cs[j], s = sn[j];
      const float ra = a * c - b * s, rb = b * c + a * s;
      a = ra;
      b = rb;
    }
    store_f<TO>(out, ia, a);
    store_f<TO>(out, ib, b);
  }
}

// One block per token: dK/dV rows of token first_token + i from the paged pool.
__global__ void __launch_bounds__(128)
    grad_gather(Geometry g, const float* __restrict__ dk_pool, const float* __restrict__ dv_pool,
                const int32_t* __restrict__ table, int64_t first_token, float* __restrict__ dk,
                float* __restrict__ dv, uint32_t* err) {
  const int i = blockIdx.x;
  const int64_t t = first_token + i;
  const int64_t p = t / g.P;
  const int r = (int)(t % g.P);
  const int phys = p < g.max_logical ? table[p] : -1;
  const int nv = g.Hkv * g.d / 4;
  float4* odk = reinterpret_cast<float4*>(dk + (size_t)i * g.Hkv * g.d);
  float4* odv = reinterpret_cast<float4*>(dv + (size_t)i * g.Hkv * g.d);
  if (phys < 0 || phys >= g.num_phys) {
    if (threadIdx.x == 0) atomicOr(err, OOMB_DEVERR_PAGE);
    for (int v = threadIdx.x; v < nv; v += blockDim.x) odk[v] = odv[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int d4 = g.d / 4;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const int h = v / d4, c = v % d4;
    const size_t src = (((size_t)phys * g.Hkv + h) * g.P + r) * g.d / 4 + c;
    odk[v] = reinterpret_cast<const float4*>(dk_pool)[src];
    odv[v] = reinterpret_cast<const float4*>(dv_pool)[src];
  }
}

template <typename TI, typename TO>
cudaError_t launch_rope(const void* in, const float* bias, void* out, int n, int H, int d, int64_t pos0,
                        float theta, int mode, cudaStream_t st) {
  bias_rope<TI, TO><<<n, kRopeThreads, 0, st>>>((const TI*)in, bias, (TO*)out, H, d, pos0,
                                                std::log2((double)theta), mode);
  count_launches(1);
  return cudaGetLastError();
}

// cuBLASLt handle per device (a host object, created on first use).
cublasLtHandle_t lt_handle(cudaError_t* e) {
  static std::mutex mu;
  static cublasLtHandle_t handles[kMaxDevices] = {};
  int dev = 0;
  *e = cudaGetDevice(&dev);
  if (*e != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *e = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!handles[dev] && cublasLtCreate(&handles[dev]) != CUBLAS_STATUS_SUCCESS) handles[dev] = nullptr;
  return handles[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace oomb

using namespace oomb;

extern "C" {

oomb_status oomb_gemm(int m, int n, int k, int trans_a, int trans_b, const void* a, const void* b, void* c,
                      int dtype_ab, int dtype_c, float alpha, float beta, void* workspace, size_t ws_bytes,
                      void* stream) {
  if (m <= 0 || n <= 0 || k <= 0 || !a || !b || !c) return OOMB_ERR_ARG;
  if ((dtype_ab != OOMB_BF16 && dtype_ab != OOMB_FP32) || (dtype_c != OOMB_BF16 && dtype_c != OOMB_FP32))
    return OOMB_ERR_DTYPE;
  if (!aligned16(a) || !aligned16(b) || !aligned16(c) || (ws_bytes && !aligned16(workspace))) return OOMB_ERR_ALIGN;
  if (ws_bytes && !workspace) return OOMB_ERR_ARG;
  cudaError_t ce;
  cublasLtHandle_t lt = lt_handle(&ce);
  if (!lt) return ce != cudaSuccess ? OOMB_ERR_CUDA : OOMB_ERR_UNSUPPORTED;
  const cudaDataType_t tab = dtype_ab == OOMB_BF16 ? CUDA_R_16BF : CUDA_R_32F;
  const cudaDataType_t tc = dtype_c == OOMB_BF16 ? CUDA_R_16BF : CUDA_R_32F;
  // Row-major C[m, n] = op(A) op(B) is column-major C^T[n, m] = op(B)^T op(A)^T: the first
  // cuBLASLt operand is B's buffer, the second A's; a row-major buffer read column-major
  // is its transpose, so an operand stored as op() wants takes no transpose.
  const cublasOperation_t op1 = trans_b ? CUBLAS_OP_T : CUBLAS_OP_N;
  const cublasOperation_t op2 = trans_a ? CUBLAS_OP_T : CUBLAS_OP_N;
  const uint64_t r1 = trans_b ? k : n, c1 = trans_b ? n : k;  // B buffer as column-major
  const uint64_t r2 = trans_a ? m : k, c2 = trans_a ? k : m;  // A buffer as column-major
  cublasLtMatmulDesc_t desc = nullptr;
  cublasLtMatrixLayout_t l1 = nullptr, l2 = nullptr, l3 = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  oomb_status st = OOMB_ERR_UNSUPPORTED;
  bool ok = cublasLtMatmulDescCreate(&desc, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatmulDescSetAttribute(desc, CUBLASLT_MATMUL_DESC_TRANSA, &op1, sizeof(op1)) ==
                CUBLAS_STATUS_SUCCESS &&
            cublasLtMatmulDescSetAttribute(desc, CUBLASLT_MATMUL_DESC_TRANSB, &op2, sizeof(op2)) ==
                CUBLAS_STATUS_SUCCESS &&
            cublasLtMatrixLayoutCreate(&l1, tab, r1, c1, (int64_t)r1) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatrixLayoutCreate(&l2, tab, r2, c2, (int64_t)r2) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatrixLayoutCreate(&l3, tc, (uint64_t)n, (uint64_t)m, (int64_t)n) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatmulPreferenceCreate(&pref) == CUBLAS_STATUS_SUCCESS &&
            cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes,
                                                 sizeof(ws_bytes)) == CUBLAS_STATUS_SUCCESS;
  if (ok) {
    cublasLtMatmulHeuristicResult_t res;
    int found = 0;
    if (cublasLtMatmulAlgoGetHeuristic(lt, desc, l1, l2, l3, l3, pref, 1, &res, &found) == CUBLAS_STATUS_SUCCESS &&
        found > 0) {
      const cublasStatus_t s = cublasLtMatmul(lt, desc, &alpha, b, l1, a, l2, &beta, c, l3, c, l3, &res.algo,
                                              workspace, ws_bytes, (cudaStream_t)stream);
      st = s == CUBLAS_STATUS_SUCCESS ? OOMB_OK : OOMB_ERR_CUDA;
    }
  }
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (l3) cublasLtMatrixLayoutDestroy(l3);
  if (l2) cublasLtMatrixLayoutDestroy(l2);
  if (l1) cublasLtMatrixLayoutDestroy(l1);
  if (desc) cublasLtMatmulDescDestroy(desc);
  return st;
}

oomb_status oomb_bias_rope(const void* in, int in_dtype, const float* bias, void* out, int out_dtype, int n, int H,
                           int d, int64_t pos0, float theta, int mode, void* stream) {
  if (!in || !out || n <= 0 || H <= 0 || d <= 0 || d % 2 || d > 2 * kMaxHalf || pos0 < 0) return OOMB_ERR_ARG;
  if (mode < 0 || mode > 2 || (mode != 0 && !(theta > 1.0f))) return OOMB_ERR_ARG;
  if ((in_dtype != OOMB_BF16 && in_dtype != OOMB_FP32) || (out_dtype != OOMB_BF16 && out_dtype != OOMB_FP32))
    return OOMB_ERR_DTYPE;
  if (in == out && in_dtype != out_dtype) return OOMB_ERR_ARG;
  // the kernel reads and writes single elements: each pointer on its element's size
  const uintptr_t ea = in_dtype == OOMB_FP32 ? 4 : 2, eb = out_dtype == OOMB_FP32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(in) % ea || reinterpret_cast<uintptr_t>(out) % eb ||
      reinterpret_cast<uintptr_t>(bias) % 4)
    return OOMB_ERR_ALIGN;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e;
  if (in_dtype == OOMB_FP32 && out_dtype == OOMB_FP32)
    e = launch_rope<float, float>(in, bias, out, n, H, d, pos0, theta, mode, st);
  else if (in_dtype == OOMB_FP32)
    e = launch_rope<float, __nv_bfloat16>(in, bias, out, n, H, d, pos0, theta, mode, st);
  else if (out_dtype == OOMB_FP32)
    e = launch_rope<__nv_bfloat16, float>(in, bias, out, n, H, d, pos0, theta, mode, st);
  else
    e = launch_rope<__nv_bfloat16, __nv_bfloat16>(in, bias, out, n, H, d, pos0, theta, mode, st);
  return e == cudaSuccess ? OOMB_OK : OOMB_ERR_CUDA;
}

}  // extern "C"

namespace oomb {
cudaError_t launch_grad_gather(const Geometry& g, const float* dk_pool, const float* dv_pool, const int32_t* table,
                               int64_t first_token, int n_tokens, float* dk, float* dv, uint32_t* err,
                               cudaStream_t st) {
  grad_gather<<<n_tokens, 128, 0, st>>>(g, dk_pool, dv_pool, table, first_token, dk, dv, err);
  count_launches(1);
  return cudaGetLastError();
}
}  // namespace oomb
