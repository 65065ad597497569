// l2_prefetch.cuh -- warming L2 with a kernel's first operand tiles while the
// kernel before it on the stream is still running.
//
// A kernel launched as a programmatic dependent may not read memory that the
// kernel before it writes until griddepcontrol.wait returns.  A prefetch into
// L2 is not such a read: it places lines in the GPU's L2, which every SM's
// writes also go through, so a line the earlier kernel writes afterwards is
// updated there and the later TMA load (issued after the wait) sees the new
// data.  Prefetching a CTA's first pipeline stages before the wait overlaps
// their DRAM latency with the earlier kernel's last microseconds.
#pragma once

#include <cstdint>

#include <cuda.h>

namespace tg {
namespace dev {

// Stages prefetched when a CTA has one tile (or one k-range) to do: deeper
// prefetches queue ahead of the real loads issued right after the wait
// (measured per call in CUDA-graph replay: the 1024 x 2048 x 512 tiling
// example 6.11 us without, 6.05 with two stages, 6.16 with all; the
// 16 x 4096 x 4096 skinny GEMM 8.97, 8.56 and 8.62 us).  A CTA with several
// tiles prefetches all its stages (256 products of 256^3: 21.3, 20.3 and
// 19.2 us).
constexpr int kPrefetchStagesSingle = 2;

// cp.async.bulk.prefetch.tensor: the box of `map` at (x, y, z) into L2, no
// shared-memory destination and no barrier.  x follows the TMA rule of the
// loads it anticipates (a multiple of 16 bytes).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int32_t x, int32_t y,
                                                   int32_t z)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// The same for a 4-D map.
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int32_t x, int32_t y,
                                                   int32_t z, int32_t w)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

}  // namespace dev
}  // namespace tg
