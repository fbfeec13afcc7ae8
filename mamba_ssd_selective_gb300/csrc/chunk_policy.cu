// Static chunk-size policy for the SSD prefill.
//
// The pages choose chunk sizes from a measured static sweep and keep the best
// per regime ("COREY ...", section 5.2: the static-oracle and learned-table
// policies, where a length-keyed table matched the per-regime oracle). This is
// that table for the bf16 tensor-core path (P = 64, N = 128) on GB300, measured
// by `python bench.py --chunk-table` over batch 1-8, sequence
// length 512-8192 and 24-80 heads; a shape off the grid takes its nearest grid
// point in (log2 batch, log2 length, heads). Shapes the tensor-core path does
// not take were not measured and get 128.
#include <cmath>
#include <cstdint>

#include "ssd_scan.h"

namespace {

struct ChunkEntry {
    int batch, seqlen, nheads, chunk;
};

// {batch, seqlen, nheads, best chunk}: measured by bench.py --chunk-table
const ChunkEntry kChunkTable[] = {
    {1, 512, 24, 64},
    {1, 1024, 24, 128},
    {1, 2048, 24, 128},
    {1, 4096, 24, 128},
    {1, 8192, 24, 128},
    {2, 512, 24, 128},
    {2, 1024, 24, 128},
    {2, 2048, 24, 128},
    {2, 4096, 24, 128},
    {2, 8192, 24, 128},
    {4, 512, 24, 128},
    {4, 1024, 24, 128},
    {4, 2048, 24, 128},
    {4, 4096, 24, 128},
    {4, 8192, 24, 128},
    {8, 512, 24, 128},
    {8, 1024, 24, 128},
    {8, 2048, 24, 128},
    {8, 4096, 24, 128},
    {8, 8192, 24, 128},
    {1, 512, 48, 128},
    {1, 1024, 48, 128},
    {1, 2048, 48, 128},
    {1, 4096, 48, 128},
    {1, 8192, 48, 128},
    {2, 512, 48, 128},
    {2, 1024, 48, 128},
    {2, 2048, 48, 128},
    {2, 4096, 48, 128},
    {2, 8192, 48, 128},
    {4, 512, 48, 128},
    {4, 1024, 48, 128},
    {4, 2048, 48, 128},
    {4, 4096, 48, 128},
    {4, 8192, 48, 128},
    {8, 512, 48, 128},
    {8, 1024, 48, 128},
    {8, 2048, 48, 128},
    {8, 4096, 48, 128},
    {8, 8192, 48, 128},
    {1, 512, 80, 128},
    {1, 1024, 80, 128},
    {1, 2048, 80, 128},
    {1, 4096, 80, 128},
    {1, 8192, 80, 128},
    {2, 512, 80, 128},
    {2, 1024, 80, 128},
    {2, 2048, 80, 128},
    {2, 4096, 80, 128},
    {2, 8192, 80, 128},
    {4, 512, 80, 128},
    {4, 1024, 80, 128},
    {4, 2048, 80, 128},
    {4, 4096, 80, 128},
    {4, 8192, 80, 128},
    {8, 512, 80, 128},
    {8, 1024, 80, 128},
    {8, 2048, 80, 128},
    {8, 4096, 80, 128},
    {8, 8192, 80, 128},
};

}  // namespace

int ssd_best_chunk(const ssd_dims *dims) {
    if (!dims) return 0;
    const ssd_dims &d = *dims;
    if (d.batch < 1 || d.seqlen < 1 || d.nheads < 1 || d.headdim < 1 || d.dstate < 1 || d.ngroups < 1 ||
        d.nheads % d.ngroups != 0 || (d.io_dtype != SSD_F32 && d.io_dtype != SSD_BF16))
        return 0;
    if (d.io_dtype != SSD_BF16 || d.headdim != 64 || d.dstate != 128) return 128;
    const double lb = std::log2((double)d.batch), ll = std::log2((double)d.seqlen);
    double best = 1e300;
    int chunk = 128;
    for (const ChunkEntry &e : kChunkTable) {
        const double db = lb - std::log2((double)e.batch), dl = ll - std::log2((double)e.seqlen);
        const double dh = ((double)d.nheads - e.nheads) / 28.0;   // 24 -> 80 heads ~ two grid steps
        const double dist = db * db + dl * dl + dh * dh;
        if (dist < best) {
            best = dist;
            chunk = e.chunk;
        }
    }
    return chunk;
}
