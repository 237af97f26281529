"""Tiling by position: a prompt's attention outputs and letter logits are bit-identical
alone, in a batch with other rows, and in a tree with sibling questions (the basal-rs
Architecture page, "05 / Reproducibility": attention tiled by position; the raw letter
scores bitwise identical alone, in a batch and in a tree)."""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import prefix_tree_packed_gb300 as lib
    return lib


def _forests(doc, q, opt, template):
    """The prompt alone: [template] -> doc -> q -> opt.  The batch: another row first, then the
    prompt's row with sibling questions and a sibling option.  Returns both forests and, for each,
    the input blocks of the prompt (root first)."""
    alone_parent, alone_len, alone_res = [], [], []
    chain = []
    for ln, res in ((template, 1), (doc, 0), (q, 0), (opt, 0)):
        if ln == 0:
            continue
        alone_parent.append(chain[-1] if chain else -1)
        alone_len.append(ln)
        alone_res.append(res)
        chain.append(len(alone_parent) - 1)
    alone = synth.Forest(np.array(alone_parent, np.int32), np.array(alone_len, np.int32),
                         np.zeros(len(alone_len), np.uint64), np.array(alone_res, np.uint8))
    par, ln_, res_ = [], [], []

    def add(p, n, r=0):
        par.append(p)
        ln_.append(n)
        res_.append(r)
        return len(par) - 1
    t = add(-1, template, 1) if template else -1
    # another row first (a different document and question)
    d2 = add(t, 333)
    q2 = add(d2, 41)
    add(q2, 17)
    add(q2, 29)
    # the prompt's row: a sibling question before and after, a sibling option before
    d = add(t, doc)
    qa = add(d, 57)
    add(qa, 11)
    qq = add(d, q)
    add(qq, 23)
    o = add(qq, opt)
    qb = add(d, 70)
    add(qb, 9)
    prompt = [x for x in (t, d, qq, o) if x >= 0]
    batch = synth.Forest(np.array(par, np.int32), np.array(ln_, np.int32), np.zeros(len(par), np.uint64),
                         np.array(res_, np.uint8))
    return alone, chain, batch, prompt


def _token_index(plan, blocks):
    """Packed token indices of the given input blocks, in order."""
    t = plan.tables()
    out = []
    for b in blocks:
        pb = t["block_map"][b]
        out += list(range(int(t["blk_start"][pb]), int(t["blk_start"][pb] + t["blk_len"][pb])))
    return np.array(out)


@pytest.mark.parametrize("d,hq,hkv,template", [(64, 4, 2, 0), (128, 4, 1, 53), (64, 32, 8, 128)])
def test_attention_bitwise_alone_batch_tree(lib, d, hq, hkv, template):
    dev = torch.device("cuda")
    alone, chain, batch, prompt = _forests(doc=300, q=50, opt=20, template=template)
    rng = np.random.default_rng(d + hq)
    n_prompt = int(sum(alone.length))
    # the prompt's own post-RoPE Q/K and V, one row per token in prompt order
    qp = rng.standard_normal((n_prompt, hq, d)).astype(np.float16)
    kp = rng.standard_normal((n_prompt, hkv, d)).astype(np.float16)
    vp = rng.standard_normal((n_prompt, hkv, d)).astype(np.float16)
    outs = {}
    pack = hq // hkv   # the q heads of a kv head in one MMA tile (tiling 1 with packed heads)
    for name, forest, blocks in (("alone", alone, chain), ("batch", batch, prompt)):
        for tiling in (0, 1, "1p"):
            plan = lib.Plan.from_forest(forest, tiling=1 if tiling == "1p" else tiling,
                                        pack_heads=pack if tiling == "1p" else 0)
            i = plan.info
            tok = _token_index(plan, blocks)
            # every other token gets its own random values
            q = rng.standard_normal((i.n_fwd, hq, d)).astype(np.float16)
            k = rng.standard_normal((i.n_tot, hkv, d)).astype(np.float16)
            v = rng.standard_normal((i.n_tot, hkv, d)).astype(np.float16)
            k[tok], v[tok] = kp, vp
            fwd = tok >= i.n_res
            q[tok[fwd] - i.n_res] = qp[fwd]
            pdev = torch.empty(i.dev_bytes, dtype=torch.uint8, device=dev)
            plan.upload(pdev, i.dev_bytes)
            o = torch.empty((i.n_fwd, hq, d), dtype=torch.float16, device=dev)
            st = torch.zeros(1, dtype=torch.int32, device=dev)
            qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, v))
            for c in range(i.n_chunks):
                ci = plan.chunk(c)
                lib.tree_attn_fwd(plan, pdev, c, qd[ci.q0 - i.n_res: ci.q1 - i.n_res], kd, vd,
                                  o[ci.q0 - i.n_res: ci.q1 - i.n_res], None, hq, hkv, d, status=st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            outs[(name, tiling)] = o.cpu().numpy()[tok[fwd] - i.n_res]
    # tiling by position: bit-identical alone and in the batch / tree
    assert np.array_equal(outs[("alone", 1)].view(np.uint16), outs[("batch", 1)].view(np.uint16))
    # alone, both tilings see the same tiles (packed index = position)
    assert np.array_equal(outs[("alone", 0)].view(np.uint16), outs[("alone", 1)].view(np.uint16))
    # with the q heads packed into the MMA tiles: the same keys in the same slots and order per row,
    # each row of an MMA tile summed on its own, so again bit-identical
    assert np.array_equal(outs[("alone", "1p")].view(np.uint16), outs[("batch", "1p")].view(np.uint16))
    assert np.array_equal(outs[("alone", "1p")].view(np.uint16), outs[("alone", 1)].view(np.uint16))


def test_model_logits_bitwise_alone_batch_tree(lib):
    """Two Llama layers (random init) ending in the letter logits: the prompt's readout row is
    bit-identical alone and in the batch with tiling by position."""
    dev = torch.device("cuda")
    alone, chain, batch, prompt = _forests(doc=300, q=50, opt=20, template=53)
    hidden, ffn, hq, hkv, d, stride, L = 256, 512, 4, 2, 64, 8, 2
    rng = np.random.default_rng(11)
    n_prompt = int(sum(alone.length))
    x_p = rng.standard_normal((n_prompt, hidden)).astype(np.float16)
    res_k = [rng.standard_normal((53, hkv * d)).astype(np.float16) for _ in range(L)]
    res_v = [rng.standard_normal((53, hkv * d)).astype(np.float16) for _ in range(L)]
    wts = [synth.draw_layer(1, 0, hidden, hq, hkv, d, ffn, 70 + l)[0] for l in range(L)]
    tds = [{k: torch.from_numpy(v).to(dev) for k, v in w.items()} for w in wts]
    layers = [lib.layer_weights(hidden, hq, hkv, d, ffn, t) for t in tds]
    wf, wl = (torch.from_numpy(a).to(dev) for a in synth.draw_head(hidden, stride, 3))
    got = {}
    for name, forest, blocks in (("alone", alone, chain), ("batch", batch, prompt)):
        plan = lib.Plan.from_forest(forest, tiling=1)
        i = plan.info
        tok = _token_index(plan, blocks)
        fwd = tok[tok >= i.n_res] - i.n_res
        x = rng.standard_normal((i.n_fwd, hidden)).astype(np.float16)
        x[fwd] = x_p[53:]
        kcs, vcs = [], []
        for l in range(L):
            kc = torch.from_numpy(rng.standard_normal((i.n_tot, hkv * d)).astype(np.float16)).to(dev)
            vc = torch.from_numpy(rng.standard_normal((i.n_tot, hkv * d)).astype(np.float16)).to(dev)
            kc[:53], vc[:53] = torch.from_numpy(res_k[l]).to(dev), torch.from_numpy(res_v[l]).to(dev)
            kcs.append(kc)
            vcs.append(vc)
        pdev = torch.empty(i.dev_bytes, dtype=torch.uint8, device=dev)
        plan.upload(pdev, i.dev_bytes)
        tab = torch.from_numpy(lib.rope_table(i.max_pos, d, 500000.0)).to(dev)
        nb = lib.model_workspace_bytes(plan, layers[0])
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        logits = torch.empty((i.n_slots, stride), device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        lib.model_fwd(plan, pdev, layers, torch.from_numpy(x).to(dev), kcs, vcs, tab, i.max_pos, wf, wl, stride,
                      logits, ws, nb, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        t = plan.tables()
        last_tok = int(tok[-1])
        slot = int(np.nonzero(t["slot_tok"] == last_tok)[0][0])
        got[name] = logits.cpu().numpy()[slot]
    assert np.array_equal(got["alone"].view(np.uint32), got["batch"].view(np.uint32))
