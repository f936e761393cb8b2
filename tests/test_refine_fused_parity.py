"""GPU parity of the fused form of selective weight refinement (StrataFlux
paper, section 3 "Weight Refinement", Eq. 2): the selections of several
activation vectors in one launch (lbq_refine_select_grouped, with the L2
prefetch of the chosen columns), then ONE grouped GEMV launch that adds each
problem's correction sum_j x_j C[:, j] to the rows it computes
(lbq_gemv_grouped_refined).  Compared with the oracle's
O.refine_apply(O.gemv(...)) element by element: both weight formats, outlier
columns, FP16 and FP32 outputs, problems without refinement in the same
launch, chunks shorter than k, and on every row of the Llama-3-8B layer
sweep; the grouped selection bit for bit against O.select_refine; and the
device-side reports of a bad index and a bad refinement header."""
import numpy as np
import pytest

from bit_weight_only_lbq_gb300 import synth
from oracle import lbq_oracle as O

from gpu_util import assert_close, to_dev
import oracle_rows

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _run(lbq, kind, specs, f32=True, seed=0):
    """specs: (N, K, n_out, k or None).  Returns [(gpu y, oracle y, gpu idx, oracle idx)]."""
    rng = np.random.default_rng(seed)
    pack, opack = (lbq.pack_w4, O.pack_w4) if kind == "w4" else (lbq.pack_w2cb, O.pack_w2cb)
    sel, probs, refs, out, keep = [], [], [], [], []
    for (N, K, n_out, k) in specs:
        W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        x = rng.standard_normal(K).astype(np.float16)
        x[rng.choice(K, size=max(1, K // 200), replace=False)] *= 100
        oidx = np.sort(rng.choice(K, size=n_out, replace=False)).astype(np.int32)
        blob = pack(W, oidx)
        y_dense = O.gemv(opack(W, oidx), x)
        dx, db = to_dev(x), to_dev(blob)
        y = torch.full((N,), float("nan"), dtype=torch.float32 if f32 else torch.float16, device="cuda:0")
        keep += [dx, db]
        probs.append((db, N, K, n_out, dx, y))
        if k is None:
            refs.append(None)
            out.append((y, y_dense, None, None))
            continue
        R = (rng.standard_normal((N, K)) * 2e-3).astype(np.float32)
        rblob = lbq.pack_refine(R)
        n_sel = lbq.refine_selected_count(K, k)
        didx = torch.full((n_sel,), -7, dtype=torch.int32, device="cuda:0")
        drb = to_dev(rblob)
        keep += [drb, didx]
        sel.append((dx, K, k, didx, drb, N))
        refs.append((drb, didx, n_sel))
        ridx = O.select_refine(x, k)
        out.append((y, O.refine_apply(rblob, x, ridx, y_dense), didx, ridx))
    lk = lbq.LBQ_KIND_W4 if kind == "w4" else lbq.LBQ_KIND_W2CB
    lbq.refine_select_grouped(sel)
    lbq.gemv_grouped_refined(lk, probs, refs, pdl=True)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    return [(y.float().cpu().numpy(), ref, None if d is None else d.cpu().numpy(), r) for y, ref, d, r in out]


# the chosen columns' pieces fit in shared memory next to the staging: they are
# copied while the weights stream
MIXED = [(64, 64, 0, 1), (320, 1088, 5, 100), (128, 2112, 0, None), (4096, 4096, 41, 16), (256, 14336, 0, 16),
         (1024, 3072, 0, 256)]
# thousands of chosen columns: the pieces do not fit, they are copied after the
# main loop into the stage ring, in batches
MANY = [(64, 8192, 64, 256), (128, 16384, 0, 256), (200 - 200 % 64, 2048, 0, 16)]


@pytest.mark.parametrize("specs", ["MIXED", "MANY"])
@pytest.mark.parametrize("kind", ["w4", "w2"])
@pytest.mark.parametrize("f32", [True, False])
def test_fused_refinement_elementwise(lbq, specs, kind, f32):
    sp = MIXED if specs == "MIXED" else MANY
    for i, (y, ref, gidx, oidx) in enumerate(_run(lbq, kind, sp, f32=f32, seed=3 if kind == "w4" else 4)):
        N, K, n_out, k = sp[i]
        if gidx is not None:
            assert np.array_equal(gidx, oidx), "grouped selection %d" % i
        assert_close(y, ref, fp16_out=not f32, what="fused refine %s %s N=%d K=%d k=%s" % (specs, kind, N, K, k))


def test_fused_refinement_llama8b_layer_every_row(lbq):
    """The bench's refined 4-bit layer sweep: the seven Llama-3-8B linears with
    C = Q4(W - W_hat), 16 channels per 1,024-channel chunk."""
    probs, refs, sel, checks, keep = [], [], [], [], []
    with oracle_rows.pool() as ex:
        for li, (name, N, K) in enumerate(synth.LLAMA3_8B_LINEARS):
            W = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA8B_W4, layer_id=li)
            x = synth.activations(1, K, workload=synth.WL_LLAMA8B_W4, layer_id=li)[0]
            blob = lbq.pack_w4(W)
            rblob = lbq.pack_refine((W - lbq.dequant_host(blob)).astype(np.float32))
            fut = oracle_rows.submit(ex, "w4", W, np.zeros(0, np.int32), x[None, :])
            del W
            n_sel = lbq.refine_selected_count(K, 16)
            dx, db, drb = to_dev(x), to_dev(blob), to_dev(rblob)
            didx = torch.empty(n_sel, dtype=torch.int32, device="cuda:0")
            y = torch.empty(N, dtype=torch.float32, device="cuda:0")
            keep += [dx, db, drb, didx]
            probs.append((db, N, K, 0, dx, y))
            sel.append((dx, K, 16, didx, drb, N))
            refs.append((drb, didx, n_sel))
            checks.append((name, y, fut, rblob, x))
        lbq.refine_select_grouped(sel)
        lbq.gemv_grouped_refined(lbq.LBQ_KIND_W4, probs, refs, pdl=True)
        torch.cuda.synchronize()
        assert lbq.device_error() == 0
        for name, y, fut, rblob, x in checks:
            ref = O.refine_apply(rblob, x, O.select_refine(x, 16), oracle_rows.collect(fut)[0])
            assert_close(y.cpu().numpy(), ref, what="refined sweep %s every row" % name)


def test_fused_refinement_reports_bad_index_and_header(lbq):
    rng = np.random.default_rng(9)
    N, K = 128, 1024
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal(K).astype(np.float16)
    rblob = lbq.pack_refine((rng.standard_normal((N, K)) * 1e-3).astype(np.float32))
    db, dx, drb = to_dev(lbq.pack_w4(W)), to_dev(x), to_dev(rblob)
    y = torch.empty(N, dtype=torch.float32, device="cuda:0")
    bad = to_dev(np.array([3, K + 5, 7], np.int32))
    lbq.gemv_grouped_refined(lbq.LBQ_KIND_W4, [(db, N, K, 0, dx, y)], [(drb, bad, 3)])
    assert lbq.device_error() == 9        # LBQ_ERR_VALUE
    wrong = rblob.copy()
    wrong[16] ^= 1                                      # N in the header
    lbq.gemv_grouped_refined(lbq.LBQ_KIND_W4, [(db, N, K, 0, dx, y)],
                             [(to_dev(wrong), to_dev(np.array([3], np.int32)), 1)])
    assert lbq.device_error() == 6        # LBQ_ERR_FORMAT
