// rpa_launch.cu -- host logic shared by rpa_forward and rpa_forward_noalloc.
//
// From a validated configuration: which kernels and tiles run (the element types decide the
// MMA operand type: bf16 for bf16 K/V, f16 for f16 and every 8-bit cache), their occupancy,
// the worst-case workspace layout, and the sequence a call enqueues on its stream:
//
//   [q conversion]  only when q's type is not the MMA operand type the kernels read (f32 q, or a
//                   16-bit q of the other 16-bit type): q rounded into the workspace
//   planner         work items, split-KV pieces, SM split
//   decode          (2-byte K/V at D 64 / 128 / 256: 8- or 16-row tiles) -- behind the prefill
//                   kernel when decode and prefill run concurrently
//   prefill         tensor-memory kernels (2-byte K/V at D 64 / 128; 8-bit K/V and 2-byte K/V at
//                   D 256, which also take the decode rows) or the latent-attention kernel (latent
//                   layout, every row)
//   combine         split-KV merge, output of the uncovered rows
//
// Each kernel is a programmatic dependent of the one before it on the caller's stream (its
// prologue overlaps the previous kernel's tail); the planner, of the previous call's combine
// kernel when that is the stream's last work.  With concurrent decode / prefill the decode
// kernel follows the prefill kernel and waits for the planner's published epoch instead of its
// grid dependency; while per-kernel profile events are on or the stream is being captured, it
// runs on the side stream instead, forked after the planner and joined before the combine.
//
// Nothing here allocates: the caller owns the workspace.
#include <string.h>

#include "rpa_internal.cuh"

namespace rpa {

namespace {

const double kLog2e = 1.4426950408889634;

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int kv_type(int32_t dt) {
    switch (dt) {
        case RPA_DT_F16: return KT_F16;
        case RPA_DT_FP8_E4M3: return KT_E4M3;
        case RPA_DT_FP8_E5M2: return KT_E5M2;
        case RPA_DT_INT8: return KT_I8;
        default: return KT_BF16;
    }
}

int out_type(int32_t dt) { return dt == RPA_DT_F32 ? OT_F32 : dt == RPA_DT_F16 ? OT_F16 : OT_BF16; }

// Byte offsets of the workspace's parts (one layout for the handle and the fixed array)
struct Layout {
    size_t ctrl, seq, units, dec, pf, comb, po, pml, qbuf, total;
};

Layout layout(const RpaCfg& c, const KernelSet& ks) {
    const int64_t S = c.max_num_seqs;
    Layout L;
    size_t off = 0;
    L.ctrl = off; off = align256(off + kCtrlWords * sizeof(int));
    L.seq = off; off = align256(off + kSeqArrays * (size_t)(S + 1) * sizeof(int));
    L.units = off; off = align256(off + (size_t)ks.max_units * 8 * sizeof(int));
    L.dec = off; off = align256(off + (size_t)ks.max_dec_units * sizeof(Unit));
    L.pf = off; off = align256(off + (size_t)ks.max_pf_units * sizeof(Unit));
    L.comb = off; off = align256(off + (size_t)ks.max_comb * sizeof(Comb));
    L.po = off; off = align256(off + (size_t)ks.max_part * kDecRows * ks.D * sizeof(float));
    L.pml = off; off = align256(off + (size_t)ks.max_part * kDecRows * 2 * sizeof(float));
    L.qbuf = off;
    if (ks.q_conv) off = align256(off + (size_t)c.num_q_tokens * c.num_q_heads * ks.D * 2);
    L.total = off;
    return L;
}

}  // namespace

void kernels_choose(const RpaCfg& c, int sms, KernelSet* ks) {
    memset(ks, 0, sizeof *ks);
    ks->G = (int)(c.num_q_heads / c.num_kv_heads);
    ks->D = (int)c.head_dim;
    ks->kt = kv_type(c.kv_dtype);
    ks->odt = out_type(c.q_dtype);
    ks->mla = c.kv_layout == RPA_KV_LATENT;
    ks->Dv = ks->mla ? (int)c.v_head_dim : ks->D;
    // the planner's head grouping: latent items hold at most 16 query rows, so a kv head's query
    // heads are planned as blocks of up to 16 ("kv heads" of the planner, reading one latent row)
    ks->Gp = ks->mla && ks->G > kMlaRows ? kMlaRows : ks->G;
    ks->Hp = (int)c.num_kv_heads * (ks->G / ks->Gp);
    const bool eight = kt_8bit(ks->kt);
    // the MMA operands of Q: bf16 with bf16 K/V, f16 otherwise; q of another type is rounded
    // into the workspace first, except bf16 q with 8-bit K/V, which the kernels round to f16 as
    // they load it
    const bool want_f16 = ks->kt != KT_BF16;
    const int qd = c.q_dtype;
    if (qd == RPA_DT_F32) {
        ks->q_conv = 1;
        ks->q_conv_f16 = want_f16;
    } else if (qd == RPA_DT_F16 && !want_f16) {
        ks->q_conv = 1;  // f16 q, bf16 K/V: q to bf16
        ks->q_conv_f16 = 0;
    } else if (qd == RPA_DT_BF16 && ks->kt == KT_F16) {
        ks->q_conv = 1;  // bf16 q, f16 K/V: q to f16
        ks->q_conv_f16 = 1;
    }
    ks->q_f16 = eight && (qd == RPA_DT_F16 || qd == RPA_DT_F32);
    const double k_sc = c.has_k_scale ? c.k_scale : 1.0;
    ks->qk_log2 = (float)(c.sm_scale * k_sc * kLog2e);
    ks->cap_exp = c.has_soft_cap ? (float)(2.0 * c.sm_scale * k_sc / c.soft_cap * kLog2e) : 0.f;
    ks->cap_log2 = c.has_soft_cap ? (float)(c.soft_cap * kLog2e) : 0.f;
    ks->v_scale = c.has_v_scale ? c.v_scale : 1.f;
    ks->window = c.has_sliding_window ? (int)(c.sliding_window > 0x7fffffff ? 0x7fffffff : c.sliding_window) : 0;
    ks->BR = 64;
    while ((int)(c.page_size % ks->BR)) ks->BR >>= 1;
    ks->br_shift = 0;
    while ((1 << ks->br_shift) < ks->BR) ++ks->br_shift;
    // 8-row decode tiles (keys on the MMA's M side) whenever a group fits: 2-byte K/V, G <= 8
    ks->dec_rows = (!eight && ks->G <= 8) ? 8 : kDecRows;
    ks->Tt = ks->G <= ks->dec_rows ? ks->dec_rows / ks->G : 1;
    ks->tc = (!ks->mla && !eight && (ks->D == 64 || ks->D == 128)) ? 1 : 0;
    // the 64-key-tile tensor-memory kernel: 8-bit K/V (converted to f16), and 2-byte K/V at D 256
    // (copied straight into its tiles)
    ks->tc8 = (!ks->mla && (eight || ks->D == 256)) ? 1 : 0;
    ks->pf_tokens = ks->tc ? 2 * (kTcRows / ks->G) : kTcRows / ks->G;
    if (ks->mla) {
        // every sequence is planned in tiles of 16 query rows; the split-KV rule takes those with
        // q_len * G' <= 16
        ks->dec_rows = kMlaRows;
        ks->Tt = kMlaRows / ks->Gp;
        ks->pf_tokens = ks->Tt;
    }
    ks->sms = sms;
}

cudaError_t kernels_occupancy(KernelSet* ks) {
    cudaError_t e = plan_prepare();
    if (e != cudaSuccess) return e;
    e = ks->mla  ? mla_prepare(ks->kt, &ks->pf_bps)
        : ks->tc ? prefill_tc_prepare(ks->D, ks->kt, &ks->pf_bps)
                 : prefill_tc8_prepare(ks->D, ks->kt, &ks->pf_bps);
    if (e != cudaSuccess) return e;
    if (ks->tc8 || ks->mla) {
        // the 8-bit tensor-memory kernel (and the latent kernel) takes the decode rows too: the
        // decode kernel never runs
        ks->dec_bps = ks->pf_bps;
    } else {
        e = decode_prepare(ks->D, ks->kt, ks->dec_rows, &ks->dec_bps);
        if (e != cudaSuccess) return e;
    }
    if (ks->pf_bps < 1 || ks->dec_bps < 1) return cudaErrorInvalidConfiguration;  // cannot be resident
    return cudaSuccess;
}

void kernels_capacity(const RpaCfg& c, KernelSet* ks) {
    // worst-case capacities (see the planner's chunk rule: at most kDecWaves pieces per CTA of
    // the kernel that runs the decode units, plus one per sequence)
    const int64_t S = c.max_num_seqs, Hkv = ks->Hp;  // the planner's kv heads
    const int64_t Tq = ks->pf_tokens;
    const int64_t dec_slots = (int64_t)ks->sms * ks->dec_bps;
    ks->max_dec_units = (int)(S + (kDecWaves * dec_slots + Hkv - 1) / Hkv + 1);
    const int pf_only_units = (int)((c.num_q_tokens + Tq - 1) / Tq + S + 1);
    ks->max_units = ks->max_dec_units + pf_only_units;
    // with 8-bit K/V on tensor memory (or latent attention), decode units are items of the
    // prefill-side kernel too
    ks->max_pf_units = (ks->tc8 || ks->mla) ? ks->max_units : pf_only_units;
    ks->max_part = (int)(ks->max_dec_units * Hkv);
    ks->max_comb = (int)(S * Hkv);
}

cudaError_t kernels_prepare(const RpaCfg& c, KernelSet* ks) {
    const cudaError_t e = kernels_occupancy(ks);
    if (e == cudaSuccess) kernels_capacity(c, ks);
    return e;
}

size_t workspace_bytes(const RpaCfg& c, const KernelSet& ks) { return layout(c, ks).total; }

Workspace workspace_carve(const RpaCfg& c, const KernelSet& ks, void* base) {
    const Layout L = layout(c, ks);
    uint8_t* b = static_cast<uint8_t*>(base);
    Workspace w;
    w.ctrl = reinterpret_cast<int*>(b + L.ctrl);
    w.seq_scratch = reinterpret_cast<int*>(b + L.seq);
    w.units = reinterpret_cast<int*>(b + L.units);
    w.dec_units = reinterpret_cast<Unit*>(b + L.dec);
    w.pf_units = reinterpret_cast<Unit*>(b + L.pf);
    w.comb = reinterpret_cast<Comb*>(b + L.comb);
    w.part_o = reinterpret_cast<float*>(b + L.po);
    w.part_ml = reinterpret_cast<float*>(b + L.pml);
    w.qbuf = ks.q_conv ? b + L.qbuf : nullptr;
    return w;
}

int enqueue_forward(const RpaCfg& c, const KernelSet& ks, const Workspace& ws, MapCache* maps, const void* q,
                    const void* kv_pages, const int32_t* kv_lens, const int32_t* page_indices,
                    const int32_t* cu_q_lens, int32_t num_seqs, void* o, const EnqueueOpts& eo) {
    cudaStream_t st = eo.st;
    const cudaEvent_t* ev = eo.ev;
    auto rec = [&](int k, cudaStream_t on) { return !ev[k] || cudaEventRecord(ev[k], on) == cudaSuccess; };
    const bool has_q = c.num_q_tokens > 0;
    if (!rec(kEvStart, st)) return RPA_ERR_CUDA;
    // q in the MMA operand type, when the caller's is another
    const void* qk = q;
    if (has_q && ks.q_conv) {
        const size_t n = (size_t)c.num_q_tokens * c.num_q_heads * ks.D;
        if (launch_q_convert(q, c.q_dtype, ws.qbuf, ks.q_conv_f16, n, Launch{ks.sms * 4, st}) != cudaSuccess)
            return RPA_ERR_CUDA;
        qk = ws.qbuf;
    }

    PlanParams pp;
    pp.kv_lens = kv_lens;
    pp.cu_q_lens = cu_q_lens;
    pp.num_seqs = num_seqs;
    pp.T = (int)c.num_q_tokens;
    pp.Hkv = ks.Hp;
    pp.G = ks.Gp;
    pp.P = (int)c.pages_per_seq;
    pp.ps = (int)c.page_size;
    pp.causal = c.is_causal ? 1 : 0;
    pp.has_window = c.has_sliding_window ? 1 : 0;
    pp.window = ks.window;
    pp.dec_rows = ks.dec_rows;
    pp.pf_tokens = ks.pf_tokens;
    pp.dec_slots = ks.sms * ks.dec_bps;
    pp.concurrent = eo.conc;
    pp.n_sms = ks.sms;
    pp.dec_bps = ks.dec_bps;
    pp.pf_bps = ks.pf_bps;
    pp.pf_mma_rows = ks.tc ? 2 * kTcRows : ks.mla ? kMlaRows : kTcRows;
    pp.dec_on_pf = ks.tc8 || ks.mla;
    pp.D = ks.D;
    pp.kv_elt = kt_8bit(ks.kt) ? 1 : 2;
    pp.pf_sm_gflops = ks.mla ? kPfSmGflopsMma : kPfSmGflopsTc;
    pp.dec_sm_gbs = kDecSmGBs;
    pp.hbm_gbs = kHbmGBs;
    pp.force_pf_sms = eo.force_pf_sms;
    pp.force_dec_sms = eo.force_dec_sms;
    pp.dec_waves = ks.tc8 ? kDecWavesTc8 : kDecWaves;
    pp.epoch = eo.epoch;
    pp.early = eo.plan_early;
    pp.max_units = ks.max_units;
    pp.max_dec_units = ks.max_dec_units;
    pp.max_pf_units = ks.max_pf_units;
    pp.max_part = ks.max_part;
    pp.max_comb = ks.max_comb;
    pp.ctrl = ws.ctrl;
    pp.seq_scratch = ws.seq_scratch;
    pp.units = ws.units;
    pp.keys = nullptr;
    pp.dec_units = ws.dec_units;
    pp.pf_units = ws.pf_units;
    pp.comb = ws.comb;
    if (launch_plan(pp, st, plan_smem_bytes()) != cudaSuccess) return RPA_ERR_CUDA;
    if (!rec(kEvPlanEnd, st)) return RPA_ERR_CUDA;

    AttnParams ap;
    ap.q = static_cast<const uint8_t*>(qk);
    ap.kv = static_cast<const uint8_t*>(kv_pages);
    ap.o = static_cast<uint8_t*>(o);
    ap.kv_lens = kv_lens;
    ap.page_indices = page_indices;
    ap.cu_q_lens = cu_q_lens;
    ap.T = (int)c.num_q_tokens;
    ap.Hq = (int)c.num_q_heads;
    ap.Hkv = (int)c.num_kv_heads;
    ap.G = ks.Gp;
    ap.D = ks.D;
    ap.ps = (int)c.page_size;
    ap.P = (int)c.pages_per_seq;
    ap.N = (int)c.total_num_pages;
    ap.causal = c.is_causal ? 1 : 0;
    ap.has_window = c.has_sliding_window ? 1 : 0;
    ap.window = ks.window;
    ap.has_cap = c.has_soft_cap ? 1 : 0;
    ap.qk_log2 = ks.qk_log2;
    ap.cap_exp = ks.cap_exp;
    ap.cap_log2 = ks.cap_log2;
    ap.v_scale = ks.v_scale;
    ap.ctrl = ws.ctrl;
    ap.units = nullptr;
    ap.unit_heads = ks.Hp;
    ap.item_count_word = 0;
    ap.counter_word = 0;
    ap.part_o = ws.part_o;
    ap.part_ml = ws.part_ml;
    ap.sinks = c.has_sinks ? c.sinks : nullptr;
    ap.odt = ks.odt;
    ap.q_f16 = ks.q_f16;

    // With the side stream forked (concurrent decode / prefill while profiling), every return
    // joins it back (st waits for whatever was enqueued there), so that no kernel of this call is
    // still writing the workspace or o when the caller's stream moves on.
    cudaStream_t dst = st;  // stream of the decode kernel
    bool forked = false;
    auto join = [&]() -> bool {
        if (!forked) return true;
        forked = false;
        return cudaEventRecord(eo.ev_dec, eo.side) == cudaSuccess && cudaStreamWaitEvent(st, eo.ev_dec, 0) == cudaSuccess;
    };
    auto fail = [&](int code) {
        join();
        return code;
    };
    // Concurrent decode / prefill on one stream: the decode kernel is launched behind the
    // prefill kernel (both programmatic dependents, so its CTAs take the SMs the prefill kernel
    // leaves) and waits for the planner's published epoch instead.  With the per-kernel profile
    // events on, the events between kernels would serialise them, and a captured graph would
    // replay one epoch: the decode kernel then runs on the side stream, forked after the planner.
    // Under stream capture (a CUDA graph replays the call's parameters, the epoch included) the
    // fork and join become graph edges instead.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (eo.conc && cudaStreamIsCapturing(st, &cap) != cudaSuccess) return RPA_ERR_CUDA;
    const bool one_stream = eo.conc && !ev[kEvStart] && cap == cudaStreamCaptureStatusNone;
    if (eo.conc && !one_stream) {
        if (cudaEventRecord(eo.ev_plan, st) != cudaSuccess || cudaStreamWaitEvent(eo.side, eo.ev_plan, 0) != cudaSuccess)
            return RPA_ERR_CUDA;
        dst = eo.side;
        forked = true;
    }
    const int byte_kv = kt_8bit(ks.kt) ? 1 : 0;
    if (has_q) {
        if (maps->kv_ptr != kv_pages) {
            if ((ks.mla ? encode_kv_map_heads(&maps->kv, kv_pages, c.total_num_pages, (int)c.page_size,
                                              (int)c.num_kv_heads, ks.D, ks.BR)
                        : encode_kv_map_runs(&maps->kv, kv_pages, byte_kv, c.total_num_pages, (int)c.page_size,
                                             (int)c.num_kv_heads, ks.D, ks.BR)) != 0 ||
                ((ks.tc || (ks.tc8 && !byte_kv)) &&
                 (tc8_whole_tiles(ks)
                      ? encode_kv_map_heads(&maps->kv_pf, kv_pages, c.total_num_pages, (int)c.page_size,
                                            2 * (int)c.num_kv_heads, ks.D, ks.BR)
                      : encode_kv_map(&maps->kv_pf, kv_pages, byte_kv, c.total_num_pages, (int)c.page_size,
                                      (int)c.num_kv_heads, ks.D, ks.BR)) != 0)) {
                maps->kv_ptr = nullptr;
                return fail(RPA_ERR_INVALID_ARG);
            }
            maps->kv_ptr = kv_pages;
        }
        if (maps->q_ptr != qk) {
            if (encode_q_map(&maps->q, qk, c.num_q_tokens, (int)c.num_q_heads, ks.D, ks.Gp, ks.Tt) != 0 ||
                ((ks.tc || ks.tc8) && encode_q_map(&maps->q_pf, qk, c.num_q_tokens, (int)c.num_q_heads, ks.D,
                                                   ks.G, kTcRows / ks.G) != 0)) {
                maps->q_ptr = nullptr;
                return fail(RPA_ERR_INVALID_ARG);
            }
            maps->q_ptr = qk;
        }
    }
    const AttnParams ap_dec = ap;
    auto launch_dec = [&](cudaStream_t on, int plan_epoch) -> bool {
        if (!rec(kEvDecStart, on)) return false;
        if (has_q && !ks.tc8 && !ks.mla) {
            DecParams dp;
            dp.a = ap_dec;
            dp.a.units = ws.dec_units;
            dp.a.item_count_word = kNumDecItems;
            dp.a.counter_word = kDecCounter;
            dp.BR = ks.BR;
            dp.br_shift = ks.br_shift;
            dp.Tt = ks.Tt;
            dp.debug_stall = eo.debug_stall;
            dp.timeout_ns = eo.timeout_ns;
            dp.plan_epoch = plan_epoch;
            if (launch_decode_tma(maps->kv, maps->q, dp, ks.kt, ks.dec_rows, Launch{ks.sms * ks.dec_bps, on}) !=
                cudaSuccess)
                return false;
        }
        return rec(kEvDecEnd, on);
    };
    if (!one_stream && !launch_dec(dst, -1)) return fail(RPA_ERR_CUDA);

    if (!rec(kEvPfStart, st)) return fail(RPA_ERR_CUDA);
    if (has_q) {
        ap.units = ws.pf_units;
        ap.item_count_word = kNumPfItems;
        ap.counter_word = kPfCounter;
        cudaError_t e;
        if (ks.mla) {
            TcParams tp;
            tp.a = ap;
            tp.BR = ks.BR;
            tp.Tq = ks.pf_tokens;
            tp.timeout_ns = eo.timeout_ns;
            e = launch_mla(maps->kv, maps->q, tp, ks.kt, Launch{ks.sms * ks.pf_bps, st});
        } else {
            TcParams tp;
            tp.a = ap;
            tp.BR = ks.BR;
            tp.Tq = ks.pf_tokens;
            tp.timeout_ns = eo.timeout_ns;
            // the 64-key-tile kernel copies whole page runs (K and V of the head) with the decode
            // gather's map for 8-bit K/V, and 128-byte column blocks with the slot x row map for 2-byte
            e = ks.tc ? launch_prefill_tc(maps->kv_pf, maps->q_pf, tp, ks.kt, Launch{ks.sms * ks.pf_bps, st})
                      : launch_prefill_tc8(byte_kv ? maps->kv : maps->kv_pf, maps->q_pf, tp, ks.kt,
                                           Launch{ks.sms * ks.pf_bps, st});
        }
        if (e != cudaSuccess) return fail(RPA_ERR_CUDA);
    }
    if (!rec(kEvPfEnd, st)) return fail(RPA_ERR_CUDA);
    if (one_stream && !launch_dec(st, eo.epoch)) return RPA_ERR_CUDA;
    if (!join()) return RPA_ERR_CUDA;

    CombParams cp;
    cp.o = static_cast<uint8_t*>(o);
    cp.cu_q_lens = cu_q_lens;
    cp.num_seqs = num_seqs;
    cp.T = (int)c.num_q_tokens;
    cp.Hq = (int)c.num_q_heads;
    cp.G = ks.Gp;
    cp.D = ks.Dv;  // the width of o and of the split-KV partials
    cp.rows_max = ks.dec_rows;
    cp.v_scale = ks.v_scale;
    cp.sinks = ap.sinks;
    cp.odt = ks.odt;
    cp.ctrl = ws.ctrl;
    cp.comb = ws.comb;
    cp.part_o = ws.part_o;
    cp.part_ml = ws.part_ml;
    if (!rec(kEvCombStart, st)) return RPA_ERR_CUDA;
    if (launch_combine(cp, Launch{ks.sms * kCombCtasPerSm, st}) != cudaSuccess) return RPA_ERR_CUDA;
    if (!rec(kEvCombEnd, st)) return RPA_ERR_CUDA;
    return RPA_OK;
}

}  // namespace rpa
