// static_scratch.cu - compiling a Command without any device allocation.
//
// Some callers cannot call cudaMalloc: programs whose device memory is owned
// entirely by their own pool or a framework's allocator (an arena sized once
// at start-up, a memory budget the CUDA allocator must not grow), where an
// allocation outside the pool is refused or breaks the accounting. cmd_compile
// allocates one small device word per kernel (the tile executor reports a
// device-side wait that ran out of time in it), so such callers use
// cmd_compile_static_scratch instead: the kernels it returns keep that word in
// the file-scope array below, which every GPU that loads this library holds
// until the process exits. Launching, status reporting and destruction are the
// usual entry points. Like cmd_compile, the call makes synchronous copies and
// may synchronise the device, so it is made outside any stream capture.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/cmd.h"
#include "cmd_internal.h"

namespace cmdx {
cmd_status compile_with_static_word(cmd_command_t cmd, cmd_kernel_t* out, uint32_t* words, int capacity);
void set_last_error(cmd_status s, const char* msg);
}  // namespace cmdx

// One error word per constant-memory program slot (kMaxPrograms = 48 are
// used): 256 bytes in all.
constexpr int kStaticWords = 64;
static_assert(cmdx::kMaxPrograms <= kStaticWords, "one static word per program slot");
static __device__ __align__(256) uint32_t g_static_scratch[kStaticWords];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_addr[kMaxDevices] = {};

}  // namespace

extern "C" cmd_status cmd_compile_static_scratch(cmd_command_t cmd, cmd_kernel_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cmdx::set_last_error(CMD_ERR_CUDA, cudaGetErrorString(e));
    return CMD_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    cmdx::set_last_error(CMD_ERR_LIMIT, "device index beyond the static scratch table");
    return CMD_ERR_LIMIT;
  }
  uint32_t* words = nullptr;
  {
    // once per device, with that device current: the array's device address
    // (the name itself is only a host-side stand-in in host code)
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess) {
        cmdx::set_last_error(CMD_ERR_CUDA, cudaGetErrorString(e));
        return CMD_ERR_CUDA;
      }
      g_addr[dev] = static_cast<uint32_t*>(p);
    }
    words = g_addr[dev];
  }
  return cmdx::compile_with_static_word(cmd, out, words, kStaticWords);
}
