// Cache-format codec: fp32 latents -> E2M1 codes with E4M3 (main KV) or E8M0
// (indexer key) group scales.  "DeepSeek-V4.1-Flash: pushing the limits of KV
// cache compression", section 5 (s_g = E4M3(max|x|/6), xhat = s_g E2M1(x/s_g));
// "DeepSeek-V4.1-Flash course, 02 Architecture", 2.4.4 (OCP MXFP4 indexer key).
#include "codec.cuh"
#include "timing.cuh"

namespace csa2 {

__global__ void k_quantize_main(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ codes,
                                uint8_t* __restrict__ scales) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n * 32) return;
  quantize_main_group(x + t * 16, codes + t * 8, scales + t);
}

__global__ void k_quantize_index(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ codes,
                                 uint8_t* __restrict__ scales) {
  int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n * 4) return;
  quantize_index_group(x + t * 32, codes + t * 16, scales + t);
}

void launch_quantize(const float* Cbar, const float* KI, int64_t n, const csa2_kv_planes* dst,
                     int64_t e0, cudaStream_t st) {
  if (n <= 0) return;
  if (Cbar) {
    int64_t threads = n * 32;
    KernelTimer timer("k_quantize_main", st);
    k_quantize_main<<<(unsigned)cdiv(threads, 256), 256, 0, st>>>(
        Cbar, n, dst->kv_codes + e0 * 256, dst->kv_scales + e0 * 32);
  }
  if (KI) {
    int64_t threads = n * 4;
    KernelTimer timer("k_quantize_index", st);
    k_quantize_index<<<(unsigned)cdiv(threads, 256), 256, 0, st>>>(
        KI, n, dst->ix_codes + e0 * 64, dst->ix_scales + e0 * 4);
  }
}

}  // namespace csa2

extern "C" csa2_status csa2_quantize_entries(const float* Cbar, const float* KI, int64_t n,
                                             const csa2_kv_planes* dst, int64_t e0,
                                             csa2_stream stream) {
  using namespace csa2;
  if (n < 0 || e0 < 0 || !planes_ok(dst)) return CSA2_ERR_INVALID_ARG;
  if ((Cbar && !aligned(Cbar, 16)) || (KI && !aligned(KI, 16))) return CSA2_ERR_INVALID_ARG;
  if (n == 0) return CSA2_OK;
  if (n > (int64_t)1 << 36) return CSA2_ERR_UNSUPPORTED;
  launch_quantize(Cbar, KI, n, dst, e0, (cudaStream_t)stream);
  return launch_status();
}
