// Decode attention without a caller-provided workspace: the split-context
// partials live in a fixed, file-scope device array instead of memory the
// caller allocates.  For callers that cannot allocate device memory when
// they run a step (see pa_paged_attention_decode_noalloc in pagedattn.h).
#include <cuda_runtime.h>

#include <mutex>

#include "pagedattn.h"

namespace {

// One scratch array per device that loads the library, held until exit.
// Host code must not take its address directly (on the host this name is
// only a stand-in for the device symbol); scratch_address() looks up the
// real device address.
__device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the first call on a device does it, with that device current).
// Under lazy module loading (the CUDA default) this lookup is also what loads
// this file's module on the device, and so what reserves the array there.
void* scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" int pa_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                                 const void* v_cache, const int32_t* block_tables,
                                                 int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                                                 int max_seq_len, int num_blocks, float scale, int num_q_heads,
                                                 int num_kv_heads, int head_dim, int block_size,
                                                 int partition_size, int dtype, void* stream) {
    if (num_seqs < 0 || max_seq_len < 0 || partition_size < 0) return PA_ERR_INVALID_ARG;
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len, partition_size);
    if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE_TOO_SMALL;
    // set-up first, even for a call with no sequences: such a call reserves
    // the array on this device and does nothing else
    void* ws = scratch_address();
    if (!ws) return PA_ERR_CUDA;
    if (num_seqs == 0) return PA_OK;
    return pa_paged_attention_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens,
                                     num_seqs, max_seq_len, num_blocks, scale, num_q_heads, num_kv_heads,
                                     head_dim, block_size, partition_size, ws, need, dtype, stream);
}
