"""Guard bands: every output buffer of the device calls sits between two
canary-filled bands, which must be intact after the call. A stand-in for a
memory checker (compute-sanitizer is not available on the GPU pool)."""
import numpy as np
import pytest
import torch

import synth
from harness import DeviceCase, make_plan
from paged_non_uniform_gb300 import kvx
import pages

pytestmark = pytest.mark.gpu
BAND = 4096  # bytes on each side


def guarded(nbytes, dtype=torch.uint8, fill=0):
    """(inner view, whole buffer): inner is nbytes (16-byte aligned) between
    two BAND-byte canary bands."""
    whole = torch.full((BAND + nbytes + BAND,), 0xA5, dtype=torch.uint8, device="cuda")
    inner = whole[BAND:BAND + nbytes]
    inner.fill_(fill)
    return inner.view(dtype), whole


def intact(whole):
    w = whole.cpu().numpy()
    return bool(np.all(w[:BAND] == 0xA5) and np.all(w[-BAND:] == 0xA5))


@pytest.mark.parametrize("kernel", [kvx.KVX_KERNEL_MMA, kvx.KVX_KERNEL_SIMT])
def test_attention_output_and_workspace_bands(kernel):
    case = synth.dense_case(2, 16, 4, 128, [700, 333], [[700, 70, 33, 1], [333, 200, 1, 64]],
                            "bf16", seed=3, P=16, head_group=[0, 1, 1, 0])
    plan = make_plan(case, num_ctas=7, kernel=kernel)
    dev = DeviceCase(case, plan)
    out, out_w = guarded(case.B * case.Hq * case.D * 4, torch.float32, 0)
    wsb = (plan.workspace_bytes() + 255) // 256 * 256
    ws, ws_w = guarded(wsb, torch.int32, 0)
    kvx.kvx_decode_attn(plan, dev.q, dev.k_pools, dev.v_pools, dev.pool_pages, dev.pt,
                        dev.strides, dev.budget, dev.seq_len, 0.0, out.view(case.B, case.Hq, -1),
                        ws, workspace_bytes=wsb)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(ws) == 0
    assert intact(out_w) and intact(ws_w)
    assert torch.isfinite(out).all()


def test_kept_row_attention_output_and_workspace_bands():
    case = synth.dense_case(2, 16, 4, 128, [700, 333], [[700, 70, 33, 1], [333, 200, 1, 64]],
                            "bf16", seed=4, P=16, head_group=[0, 1, 1, 0])
    plan = make_plan(case, num_ctas=7)
    conv = lambda a: torch.from_numpy(synth.f32_to_bf16_bits(a).view(np.int16)).view(
        torch.bfloat16).cuda()
    Lmax = case.k.shape[2]
    stride = max(len(x) for x in case.kept)
    kept = np.full((len(case.kept), stride), -1, np.int32)
    for i, x in enumerate(case.kept):
        kept[i, :len(x)] = x
    out, out_w = guarded(case.B * case.Hq * case.D * 4, torch.float32, 0)
    wsb = (plan.workspace_bytes() + 255) // 256 * 256
    ws, ws_w = guarded(wsb, torch.int32, 0)
    kvx.kvx_decode_attn_kept(plan, conv(case.q), conv(case.k), conv(case.v), Lmax,
                             torch.from_numpy(kept).cuda(), stride,
                             torch.from_numpy(case.budget.reshape(-1).astype(np.int32)).cuda(),
                             torch.from_numpy(case.seq_len.astype(np.int32)).cuda(), 0.0,
                             out.view(case.B, case.Hq, -1), ws, workspace_bytes=wsb)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(ws) == 0
    assert intact(out_w) and intact(ws_w)
    assert torch.isfinite(out).all()


def test_gather_staging_and_workspace_bands():
    cfg = synth.gather_config(seed=4, S=10, Lmin=1, Lmax=640, token_bytes=4, num_phys=2048,
                              extents=True, max_extent=6)
    pool = torch.from_numpy(synth.block_stamp_pool(cfg.num_phys, cfg.block_bytes, 1)).cuda()
    st, st_w = guarded(cfg.S * cfg.row_bytes)
    wsb = (kvx.kvx_gather_workspace_bytes(cfg.S, cfg.max_blocks) + 255) // 256 * 256
    ws, ws_w = guarded(wsb, torch.int32)
    kvx.kvx_gather_coalesce(torch.from_numpy(cfg.bt).cuda(), torch.from_numpy(cfg.nb).cuda(),
                            cfg.S, cfg.max_blocks, [pool], cfg.num_phys, cfg.block_bytes, [st],
                            cfg.row_bytes, kvx.KVX_ZERO_TAIL, ws, workspace_bytes=wsb)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(ws) == 0
    assert intact(st_w) and intact(ws_w)


def test_select_and_pack_bands():
    g = synth.rng(8)
    B, Hq, Hkv, D, L = 2, 8, 2, 128, np.array([1500, 777], np.int32)
    top, recent = 100, 12
    keys = synth.normal(g, (B, Hkv, 1500, D), "bf16")
    q = synth.normal(g, (B, Hq, D), "bf16")
    bf = lambda a: torch.from_numpy(synth.f32_to_bf16_bits(a).view(np.int16)).view(
        torch.bfloat16).cuda()
    kd = bf(keys)
    kept, kept_w = guarded(B * Hkv * (top + recent) * 4, torch.int32)
    cnt, cnt_w = guarded(B * Hkv * 4, torch.int32)
    wsb = (kvx.kvx_select_workspace_bytes(B, Hkv, 1500) + 255) // 256 * 256
    ws, ws_w = guarded(wsb, torch.int32)
    kvx.kvx_select_topk(kd, bf(q), torch.from_numpy(L).cuda(), B, Hq, Hkv, D, 1500, top, recent,
                        kept, cnt, ws, workspace_bytes=wsb)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(ws) == 0
    assert intact(kept_w) and intact(cnt_w) and intact(ws_w)
    n = cnt.cpu().numpy().reshape(B, Hkv)
    hg = np.zeros(Hkv, np.int32)
    plan = kvx.kvx_plan_create(B, Hq, Hkv, D, 16, 1, kvx.KVX_BF16, n, L, hg, 5)
    kvx.kvx_plan_upload(plan)
    gp = plan.group_pages()
    tables, npages = pages.assign_pages(gp, [synth.page_permutation(3, int(gp[0].sum()) + 1)], 1)
    nel = npages[0] * Hkv * 16 * D
    kp, kp_w = guarded(nel * 2, torch.bfloat16)
    vp, vp_w = guarded(nel * 2, torch.bfloat16)
    wsa = (plan.workspace_bytes() + 255) // 256 * 256
    aws, aws_w = guarded(wsa, torch.int32)
    kvx.kvx_pack_kept(plan, kd, kd, 1500, kept, top + recent, [kp], [vp], npages,
                      [torch.from_numpy(tables[0]).cuda()], [tables[0].shape[1]], aws,
                      workspace_bytes=wsa)
    torch.cuda.synchronize()
    assert kvx.kvx_workspace_status(aws) == 0
    assert intact(kp_w) and intact(vp_w) and intact(aws_w)
