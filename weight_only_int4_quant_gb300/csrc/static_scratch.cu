// Loop-block entry point that allocates nothing and needs no caller scratch.
//
// Some callers cannot provide device scratch or call cudaMalloc: a runtime
// that forbids allocation once it is serving (fixed memory budget, no
// allocator on the request path), a plugin slot in a host framework that only
// hands the layer its input and output tensors, or code that must not touch
// the allocator at all.  For them the four FP16 intermediates of the loop
// block (norm output, QKV, O and UP activations) live in one static device
// array of this file instead of caller-owned buffers, and the GEMMs run
// without the prefill kernel's k split (which needs a workspace).
#include <mutex>

#include "common.cuh"

namespace {

// Upper bound of the static scratch: every GPU that loads the library keeps
// this much device memory until the process exits.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_block_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

}  // namespace

extern "C" tlq_status tl_loop_block_forward_static_scratch(float* x, const tl_block* block, int L, int M,
                                                           void* stream) {
  using tlq::set_error;
  tlq::clear_error();
  if (!x || !block) return set_error(TLQ_EINVAL, "tl_loop_block_forward_static_scratch: null x or block");
  if (M < 1) return set_error(TLQ_EINVAL, "tl_loop_block_forward_static_scratch: M=%d (must be >= 1)", M);
  const int D = block->D, F = block->up.N;
  if (D < 1 || F < 1)
    return set_error(TLQ_EINVAL, "tl_loop_block_forward_static_scratch: D=%d F=%d must be >= 1", D, F);
  const size_t hb = round256((size_t)M * D * 2), qb = round256((size_t)M * 3 * D * 2), ob = hb,
               ub = round256((size_t)M * F * 2);
  const size_t need = hb + qb + ob + ub;
  if (need > kStaticScratchBytes)
    return set_error(TLQ_EINVAL,
                     "tl_loop_block_forward_static_scratch: M=%d, D=%d, F=%d needs %zu bytes of scratch; the "
                     "static scratch holds %zu bytes (use tl_loop_block_forward with caller buffers)",
                     M, D, F, need, kStaticScratchBytes);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tlq::cuda_error(e, "tl_loop_block_forward_static_scratch: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(TLQ_EUNSUPPORTED, "tl_loop_block_forward_static_scratch: device %d out of range", dev);
  uint8_t* base = nullptr;
  {
    // once per device, with that device current: the device address of the
    // array (its name in host code is only a stand-in for the symbol)
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_block_scratch);
      if (e != cudaSuccess) return tlq::cuda_error(e, "tl_loop_block_forward_static_scratch: cudaGetSymbolAddress");
      g_scratch_ptr[dev] = p;
    }
    base = static_cast<uint8_t*>(g_scratch_ptr[dev]);
  }
  tl_block b = *block;
  b.h = reinterpret_cast<uint16_t*>(base);
  b.qkv_out = reinterpret_cast<uint16_t*>(base + hb);
  b.o_out = reinterpret_cast<uint16_t*>(base + hb + qb);
  b.up_out = reinterpret_cast<uint16_t*>(base + hb + qb + ob);
  b.workspace = nullptr;  // no k split: that would need a workspace
  b.workspace_bytes = 0;
  return tlq::loop_block_forward_named(x, &b, L, M, "tl_loop_block_forward_static_scratch", stream);
}
