// zccl_plan.cu -- the reduce-scatter switcher's time model (host only).
//
// Page: "ZipCCL: Efficient Lossless Data Compression of Communication
// Collectives for Accelerating LLM Training", technical summary 2.D: the
// switcher profiles bandwidth, latency and the compression ratio at start-up
// and picks the native reduce-scatter or a zipped all-to-all followed by a
// local decompress-and-reduce.  The model compares the two paths' times;
// every term is a message or a codec pass, with the codec's measured rate.
#include <cmath>
#include <cstdint>

#include "../../include/zccl.h"

namespace {

bool finite_at_least(double v, double lo) { return std::isfinite(v) && v >= lo; }
bool finite_positive(double v) { return std::isfinite(v) && v > 0.0; }

// microseconds to move `bytes` at `gbs` GB/s
double transfer_us(double bytes, double gbs) { return bytes / (gbs * 1e3); }

}  // namespace

extern "C" zccl_status_t zccl_rs_plan(const zccl_rs_model_t* m, zccl_rs_plan_t* plan)
{
    if (m == nullptr || plan == nullptr || m->ranks < 1 || !finite_positive(m->ratio) ||
        !finite_positive(m->link_gbs) || !finite_at_least(m->link_latency_us, 0.0) ||
        !finite_positive(m->compress_gbs) || !finite_at_least(m->compress_fixed_us, 0.0) ||
        !finite_positive(m->reduce_gbs) || !finite_at_least(m->reduce_fixed_us, 0.0))
        return ZCCL_ERR_INVALID_ARG;
    *plan = zccl_rs_plan_t{};
    if (m->ranks == 1) return ZCCL_OK;  // one rank: nothing crosses a link

    const double peers = (double)(m->ranks - 1);
    const double shard = (double)m->bytes / (double)m->ranks;
    // both paths send one message per peer; they differ in the bytes each
    // message carries and in the codec passes the zipped path adds
    const double messages_us = peers * m->link_latency_us;
    const double raw_link_us = peers * transfer_us(shard, m->link_gbs);
    const double codec_us = m->compress_fixed_us + transfer_us(peers * shard, m->compress_gbs) +
                            m->reduce_fixed_us + transfer_us((double)m->ranks * shard, m->reduce_gbs);
    plan->native_us = messages_us + raw_link_us;
    plan->zipped_us = codec_us + messages_us + m->ratio * raw_link_us;
    plan->zipped = plan->zipped_us < plan->native_us ? 1 : 0;
    // zipped wins iff link time saved, peers * shard * (1 - ratio) / link,
    // exceeds codec_us: solve for the link bandwidth
    if (m->ratio < 1.0)
        plan->breakeven_link_gbs = codec_us > 0.0 ? peers * shard * (1.0 - m->ratio) / (codec_us * 1e3) : INFINITY;
    return ZCCL_OK;
}
