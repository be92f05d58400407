// Device-side fill of synthetic K/V blocks with the counter-based normal
// generator of sfi_workloads (SplitMix64 words + Box-Muller in fp64, rounded
// fp64 -> fp32 -> bf16 with round-to-nearest-even).  This produces the same
// bits as the numpy generator (up to last-ulp differences of the fp64 log,
// sin and cos between the two math libraries), so the very large workloads
// need not be generated on the host.  Inputs only: no method arithmetic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kPhi = 0x9E3779B97F4A7C15ULL;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__device__ __forceinline__ double normal_at(uint64_t key, uint64_t e) {
  const uint64_t p = e >> 1;
  const uint64_t w1 = mix64(key + (2 * p + 1) * kPhi);
  const uint64_t w2 = mix64(key + (2 * p + 2) * kPhi);
  const double u1 = (double(w1 >> 11) + 0.5) * 0x1.0p-53;
  const double u2 = double(w2 >> 11) * 0x1.0p-53;
  const double rad = sqrt(-2.0 * log(u1));
  const double th = 6.283185307179586 * u2;
  return (e & 1) ? rad * sin(th) : rad * cos(th);
}

// dst[i] = round(normal(key, start + i) + add[j]) for i < count, where
// j = (start + i) % d and add is applied when `rows_mask` is NULL or
// rows_mask[((start + i) / d) % cap] != 0 (add may be NULL: nothing added).
__global__ void fill_kernel(void* dst, int dtype, uint64_t key, int64_t start, int64_t count,
                            int d, int cap, const uint8_t* rows_mask, const double* add) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < count;
       i += int64_t(gridDim.x) * blockDim.x) {
    const uint64_t e = uint64_t(start + i);
    double z = normal_at(key, e);
    if (add) {
      const int j = int(e % uint64_t(d));
      const int64_t row = int64_t((e / uint64_t(d)) % uint64_t(cap));
      if (!rows_mask || rows_mask[row]) z = z + add[j];
    }
    const float f = __double2float_rn(z);
    if (dtype == 0) {
      static_cast<float*>(dst)[i] = f;
    } else {
      static_cast<__nv_bfloat16*>(dst)[i] = __float2bfloat16_rn(f);
    }
  }
}

// Row r of dst (row_len elements) is stream keys[r] at elements [0, row_len),
// plus add[j] (j = element % d) when add is not NULL.
__global__ void fill_rows_kernel(void* dst, int dtype, const uint64_t* keys, int64_t rows,
                                 int64_t row_len, int d, const double* add) {
  const int64_t count = rows * row_len;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < count;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / row_len;
    const uint64_t e = uint64_t(i - r * row_len);
    double z = normal_at(keys[r], e);
    if (add) z = z + add[int(e % uint64_t(d))];
    const float f = __double2float_rn(z);
    if (dtype == 0) {
      static_cast<float*>(dst)[i] = f;
    } else {
      static_cast<__nv_bfloat16*>(dst)[i] = __float2bfloat16_rn(f);
    }
  }
}

}  // namespace

extern "C" int sfigen_fill_rows(void* dst, int dtype, const uint64_t* keys, int64_t rows,
                                int64_t row_len, int d, const double* add, void* stream) {
  if (!dst || !keys || rows < 0 || row_len < 1 || d < 1) return 1;
  if (rows == 0) return 0;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (rows * row_len + 255) / 256;
  if (blocks > int64_t(sms) * 16) blocks = int64_t(sms) * 16;
  fill_rows_kernel<<<int(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(dst, dtype, keys, rows,
                                                                             row_len, d, add);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

extern "C" int sfigen_fill(void* dst, int dtype, uint64_t key, int64_t start, int64_t count, int d,
                           int cap, const uint8_t* rows_mask, const double* add, void* stream) {
  if (!dst || count < 0 || d < 1 || cap < 1) return 1;
  if (count == 0) return 0;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (count + 255) / 256;
  if (blocks > int64_t(sms) * 16) blocks = int64_t(sms) * 16;
  fill_kernel<<<int(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(dst, dtype, key, start,
                                                                          count, d, cap, rows_mask,
                                                                          add);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
