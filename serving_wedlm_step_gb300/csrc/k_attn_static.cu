// Paged causal window attention for callers that cannot allocate device
// memory: everything the kernels need beyond the caller's inputs and
// outputs lives in one file-scope device array (kAttnStaticScratchBytes),
// which every GPU that loads this library holds until the process exits.
//
// The host never dereferences the array's name (in host code it is only a
// stand-in); the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and then passed to the
// kernels.
#include <mutex>

#include "internal.h"

namespace wedlm {

namespace {
constexpr size_t kAttnStaticScratchBytes = (size_t)16 << 20;  // 16 MiB
constexpr size_t kErrOff = 0;         // device error word (256 B)
constexpr size_t kZeroOff = 256;      // zero page (4 KiB)
constexpr size_t kPartOff = 256 + 4096;
constexpr int kMaxDevices = 64;
}  // namespace

static __device__ __align__(256) uint8_t g_attn_scratch[kAttnStaticScratchBytes];

namespace {
std::mutex g_mu;
uint8_t* g_addr[kMaxDevices] = {};

// device address of the scratch array on the current device (set up once)
int scratch_for_current_device(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return WEDLM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return WEDLM_ERR_CUDA;
    // the zero page must hold zeros; nothing ever writes it afterwards
    if (cudaMemset(static_cast<uint8_t*>(p) + kZeroOff, 0, 4096) != cudaSuccess)
      return WEDLM_ERR_CUDA;
    g_addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_addr[dev];
  return WEDLM_OK;
}
}  // namespace

}  // namespace wedlm

using namespace wedlm;

extern "C" int wedlm_attention_static(int32_t batch, int32_t window, int32_t n_q_heads,
                                      int32_t n_kv_heads, int32_t max_pages_per_seq,
                                      int32_t num_pages, const void* q, const void* kv_pool,
                                      const int32_t* page_table, const int32_t* seq_len,
                                      const void* kv_win, void* o, void* stream) {
  const int hd = 128;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; };
  if (batch < 1 || window < 1 || window > kMaxWindow || n_kv_heads < 1 ||
      n_q_heads < n_kv_heads || n_q_heads % n_kv_heads ||
      (n_q_heads / n_kv_heads) * window > 128 || max_pages_per_seq < 1 || num_pages < 1 ||
      !q || !kv_pool || !page_table || !seq_len || !kv_win || !o || misaligned(q) ||
      misaligned(kv_pool) || misaligned(kv_win) || misaligned(o))
    return WEDLM_ERR_INVALID_ARG;
  const int Wp = ((window + kPageBlock - 1) / kPageBlock) * kPageBlock;
  const int R = (n_q_heads / n_kv_heads) * window;
  if (Wp > 64 || batch * window > kMaxRows) return WEDLM_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms < 1)
    return WEDLM_ERR_CUDA;
  // segment counts + partials of at most (blocks + units) segments of R rows
  const size_t units = (size_t)batch * n_kv_heads;
  const size_t table_bytes = ((units * sizeof(int) + 255) / 256) * 256;
  const size_t slots = (size_t)sms + units;
  const size_t need = kPartOff + table_bytes + slots * R * (hd + 2) * sizeof(float);
  if (need > kAttnStaticScratchBytes) return WEDLM_ERR_CAPACITY;  // beyond the array

  uint8_t* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch + kErrOff, 0, 4, st) != cudaSuccess) return WEDLM_ERR_CUDA;
  int* unit_cnt = reinterpret_cast<int*>(scratch + kPartOff);
  // the kernel leaves the counts at zero; clearing them here as well keeps a
  // call that gave up on a wait from leaking counts into the next one
  if (cudaMemsetAsync(unit_cnt, 0, units * sizeof(int), st) != cudaSuccess) return WEDLM_ERR_CUDA;
  float* part_o = reinterpret_cast<float*>(scratch + kPartOff + table_bytes);
  float* part_ml = part_o + slots * R * hd;

  AttnArgs A{};
  A.B = batch; A.W = window; A.Wp = Wp; A.nq = n_q_heads; A.nkv = n_kv_heads; A.hd = hd;
  A.num_pages = num_pages; A.max_pages = max_pages_per_seq; A.pt_stride = max_pages_per_seq;
  A.scale_log2 = (float)(1.4426950408889634 / 11.313708498984761);  // log2(e)/sqrt(128)
  A.q = q; A.pool = kv_pool; A.page_table = page_table; A.seq_len = seq_len;
  A.kv_win = kv_win; A.part_o = part_o; A.part_ml = part_ml; A.o = o;
  A.err = reinterpret_cast<int*>(scratch + kErrOff);
  A.min_tiles = 2;
  A.unit_cost = kAttnUnitCost;  // the same split as wedlm_attention
  A.unit_cnt = unit_cnt;
  if (launch_attention_tc(A, scratch + kZeroOff, sms, st) != cudaSuccess) return WEDLM_ERR_CUDA;
  return WEDLM_OK;
}

extern "C" int wedlm_attention_static_status(void* stream, int32_t* device_error) {
  if (!device_error) return WEDLM_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return WEDLM_ERR_CUDA;
  uint8_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    scratch = g_addr[dev];
  }
  int32_t word = 0;
  if (scratch) {  // else no call has run on this device
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&word, scratch + kErrOff, sizeof(word), cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return WEDLM_ERR_CUDA;
  }
  *device_error = word;
  return WEDLM_OK;
}
