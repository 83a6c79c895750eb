// Host-side plumbing of libte_gb300: status strings, the asynchronous error
// word, launch accounting, tensor-map encoding and the block-scale layout helpers.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace {

// Device error word: kernels whose bounded waits expire write TE_ERR_TIMEOUT here.
__device__ int g_device_error_word;

std::atomic<int> g_host_error{0};
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {nullptr};
int g_sms[kMaxDevices] = {0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return (d >= 0 && d < kMaxDevices) ? d : 0;
}

// One warp waits on a barrier that nothing completes: the bounded wait gives up
// after ~10 ms, records TE_ERR_TIMEOUT and the kernel returns normally.
__global__ void selftest_wait_kernel(int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    te::dev::mbar_init(&bar, 1);
    abort_flag = 0;
    te::dev::fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) te::dev::mbar_wait_limit(&bar, 0, &abort_flag, err, 20000000LL);
  __syncwarp();
}

}  // namespace

namespace te {

te_status record_cuda(cudaError_t e) {
  if (e == cudaSuccess) return TE_OK;
  int expected = 0;
  g_host_error.compare_exchange_strong(expected, static_cast<int>(TE_ERR_CUDA));
  return TE_ERR_CUDA;
}

void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }

int* device_error_word() {
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_err_ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<int*>(p);
  }
  return g_err_ptr[d];
}

int num_sms() {
  const int d = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[d] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 1;
  }
  return g_sms[d];
}

static te_status encode_2d_typed(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t elem_bytes,
                                 uint64_t cols, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
                                 CUtensorMapSwizzle swz) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return record_cuda(cudaErrorInitializationError);
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return record_cuda(cudaErrorInvalidValue);
  return TE_OK;
}

static te_status encode_2d(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_inner,
                           uint32_t box_rows, CUtensorMapSwizzle swz) {
  return encode_2d_typed(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, row_bytes, rows, box_inner, box_rows, swz);
}

te_status make_tmap_2d(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
  return encode_2d(map, base, row_bytes, rows, 128u, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

te_status make_tmap_2d_plain(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows,
                             uint32_t box_inner_bytes, uint32_t box_rows) {
  return encode_2d(map, base, row_bytes, rows, box_inner_bytes, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

te_status make_tmap_2d_f32(CUtensorMap* map, const float* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                           uint32_t box_rows) {
  return encode_2d_typed(map, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, cols, rows, box_cols, box_rows,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
}

te_status make_tmap_2d_boxswz(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows,
                              uint32_t box_inner_bytes, uint32_t box_rows) {
  const CUtensorMapSwizzle swz = box_inner_bytes == 64   ? CU_TENSOR_MAP_SWIZZLE_64B
                                 : box_inner_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                         : CU_TENSOR_MAP_SWIZZLE_NONE;
  return encode_2d(map, base, row_bytes, rows, box_inner_bytes, box_rows, swz);
}

}  // namespace te

namespace {

bool scale_geometry(te_dtype fmt, int64_t rows, int64_t cols, int64_t* block, int64_t* rpad, int64_t* kpad) {
  if (rows < 0 || cols < 0) return false;
  if (fmt == TE_E8M0) {
    *block = 32;
    if (cols % 32) return false;
    *kpad = ((cols / 32 + 3) / 4) * 4;
  } else if (fmt == TE_UE4M3) {
    *block = 16;
    if (cols % 16) return false;
    *kpad = ((cols / 16 + 15) / 16) * 16;
  } else {
    return false;
  }
  *rpad = ((rows + 127) / 128) * 128;
  return true;
}

}  // namespace

extern "C" {

size_t te_scale_bytes(te_dtype scale_fmt, int64_t rows, int64_t cols) {
  int64_t blk, rpad, kpad;
  if (!scale_geometry(scale_fmt, rows, cols, &blk, &rpad, &kpad)) return 0;
  return static_cast<size_t>(rpad * kpad);
}

te_status te_scale_unswizzle(te_dtype scale_fmt, int64_t rows, int64_t cols, const uint8_t* swizzled,
                             uint8_t* logical) {
  int64_t blk, rpad, kpad;
  if (!scale_geometry(scale_fmt, rows, cols, &blk, &rpad, &kpad)) return TE_ERR_SHAPE;
  if ((swizzled == nullptr || logical == nullptr) && rows * cols > 0) return TE_ERR_NULL;
  const int64_t nb = cols / blk;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t j = 0; j < nb; ++j)
      logical[r * nb + j] = swizzled[te::scale_offset(static_cast<uint64_t>(r), static_cast<uint64_t>(j),
                                                      static_cast<uint64_t>(kpad))];
  return TE_OK;
}

const char* te_status_str(te_status s) {
  switch (s) {
    case TE_OK: return "TE_OK";
    case TE_ERR_NULL: return "TE_ERR_NULL: required pointer is NULL";
    case TE_ERR_SHAPE: return "TE_ERR_SHAPE: dimension violates the call's constraints";
    case TE_ERR_ALIGN: return "TE_ERR_ALIGN: pointer not 16-byte aligned";
    case TE_ERR_DTYPE: return "TE_ERR_DTYPE: dtype not accepted";
    case TE_ERR_UNSUPPORTED: return "TE_ERR_UNSUPPORTED: combination not implemented";
    case TE_ERR_CUDA: return "TE_ERR_CUDA: CUDA runtime failure";
    case TE_ERR_TIMEOUT: return "TE_ERR_TIMEOUT: device-side wait gave up";
    case TE_ERR_ARG: return "TE_ERR_ARG: invalid argument";
  }
  return "unknown te_status";
}

te_status te_get_last_error(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) te::record_cuda(e);
  int* p = te::device_error_word();
  if (p != nullptr) {
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess && v != 0) {
      int zero = 0;
      cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
      int expected = 0;
      g_host_error.compare_exchange_strong(expected, v);
    }
  }
  int h = g_host_error.exchange(0);
  return static_cast<te_status>(h);
}

uint64_t te_launch_count(void) { return g_launches.load(); }

te_status te_selftest_wait_timeout(void* stream) {
  int* err = te::device_error_word();
  if (err == nullptr) return te::record_cuda(cudaErrorInvalidDevice);
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err);
  te::count_launch();
  return te::launch_status();
}

}  // extern "C"
