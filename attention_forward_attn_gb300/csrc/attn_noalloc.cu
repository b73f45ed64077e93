// attn_fwd_noalloc: the attention forward for callers that must not allocate
// device memory.
//
// attn_fwd needs one word of device scratch memory -- the device status word
// its kernel writes when a bounded wait gives up or a valid_len value is
// clamped -- and allocates it with cudaMalloc on its first call on a device.
// Some callers cannot let a library do that: servers that reserve all device
// memory at start-up and forbid allocations on the request path (cudaMalloc
// can synchronise the device and stall every other stream), latency-bound
// loops that cannot afford an allocation's unpredictable cost, and embedders
// whose memory accounting sees only their own allocator.  This entry point
// runs the same kernel with its scratch taken from a fixed array in this
// file's static device memory instead.
//
// The array is created when the CUDA module of libattn.so is loaded on a
// device and stays there until the process exits (kNoallocScratchWords
// 32-bit words, 256 bytes, on every device that loads the library).  Host code
// cannot name it as a device address: its device address is looked up once
// per device with cudaGetSymbolAddress, with that device current, on the
// first call of attn_fwd_noalloc on that device.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace {

constexpr int kNoallocScratchWords = 64;   // capacity of the static array (256 bytes)
constexpr int kStatusWordsPerCall = 1;     // what one call uses: the kernel's status word
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int g_noalloc_scratch[kNoallocScratchWords];

struct NoallocDevice {
  bool ready = false;    // set-up done on this device
  bool used = false;     // at least one call was queued (attn_status then reads the word)
  int num_sms = 0;
  int* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_mu;
NoallocDevice g_dev[kMaxDevices];

// Scratch words one call needs.  The kernel's only scratch is its status word,
// so every valid problem fits; the check keeps the array from being overrun.
int scratch_words_needed() { return kStatusWordsPerCall; }

// First call on the current device: check the architecture and look up the
// device address of the static array (no allocation).
attn_status_t setup_device(int dev, NoallocDevice** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  NoallocDevice& d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return attn::cuda_fail(e);
    if (!(prop.major == 10 && prop.minor == 3)) return ATTN_ERR_ARCH;
    int* ptr = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch);
    if (e != cudaSuccess) return attn::cuda_fail(e);
    d.num_sms = prop.multiProcessorCount;
    d.scratch = ptr;
    d.ready = true;
  }
  *out = &d;
  return ATTN_OK;
}

}  // namespace

namespace attn {

// Called by attn_status (after it synchronised): read and clear the status
// word of the no-alloc path on `dev`, if that path was ever used there.
attn_status_t noalloc_take_status(int dev, int* code) {
  if (dev < 0 || dev >= kMaxDevices) return ATTN_OK;
  int* word = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_dev[dev].used) word = g_dev[dev].scratch;
  }
  if (word == nullptr) return ATTN_OK;
  int v = 0;
  cudaError_t e = cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v != 0) {
    e = cudaMemset(word, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  *code |= v;
  return ATTN_OK;
}

}  // namespace attn

extern "C" attn_status_t attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                                          float* lse, int B, int Hq, int Hkv, int L, int D,
                                          float sm_scale, int causal, const int32_t* valid_len,
                                          attn_dtype_t dtype, attn_stream_t stream) {
  attn_status_t s =
      attn::validate(q, k, v, o, lse, B, Hq, Hkv, L, D, sm_scale, causal, valid_len, dtype);
  if (s != ATTN_OK) return s;
  if (scratch_words_needed() > kNoallocScratchWords) return ATTN_ERR_SCRATCH;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn::cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_ARCH;
  NoallocDevice* d = nullptr;
  if ((s = setup_device(dev, &d)) != ATTN_OK) return s;
  if ((s = attn::tensor_map_encoder_ready()) != ATTN_OK) return s;
  attn::Problem p = attn::make_problem(q, k, v, o, lse, B, Hq, Hkv, L, D, sm_scale, causal,
                                       valid_len, dtype, stream, d->scratch);
  // no fp16 copy of V without a workspace: bf16 tiles all take the split
  // P.V (Problem::vflags stays null); the fourth map is never read
  CUtensorMap maps[5];
  if ((s = attn::encode_problem_maps(p, maps)) != ATTN_OK) return s;
  // The status word is not cleared here: it started at zero when the module
  // was loaded, the kernel only ORs conditions into it, and attn_status
  // clears it after reading -- so, as attn_fwd's word does, it keeps every
  // condition until attn_status reads it.
  e = attn::launch_tc(p, maps, d->num_sms);
  if (e != cudaSuccess) return attn::cuda_fail(e);
  {
    std::lock_guard<std::mutex> lock(g_mu);
    d->used = true;
  }
  return ATTN_OK;
}
