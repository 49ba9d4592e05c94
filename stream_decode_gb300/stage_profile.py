"""Per-stage timeline of the cluster step kernel, from its timing hook.

    python -m stream_decode_gb300.stage_profile [--quant f32|f16] [--positions 16,64,120]

Runs the GPT-2 124M decode workload (a 16-token prompt, then greedy steps up
to position 127) and, for a run starting at each given position, records
step 0's stamps (gpt2_session_set_timing: per CTA and layer, the
globaltimer when each stage of the layer ended).  Prints the step time of
the run, and per stage the mean over layers 1..L-1 of the latest CTA's end
relative to the previous layer's end, the spread of the stage's end over
CTAs, and the vocabulary stage.  Synthetic seeded weights and tokens.
"""
import argparse

import numpy as np

STAGES = ["in", "qkvpart", "qkvgath", "attn", "ogath", "opub", "resid", "fcpart", "ugath", "mlppub"]
PROMPT, LAST = 16, 128


def profile(quant: str = "f32", positions=(16, 64, 120)):
    import torch
    from stream_decode_gb300 import gpt2 as g, synth
    shape = synth.GPT2_124M
    w = synth.checkpoint(shape, synth.SEED_124M)
    model = g.Model(shape, w, quant={"f32": g.F32, "f16": g.F16}[quant])
    kind, nc, cs = model.step_kernel
    if kind != "cluster":
        raise SystemExit("the model does not run on the cluster step kernel (GPT2_STEP_KERNEL=phase?)")
    G, L, V = nc * cs, shape.n_layer, shape.vocab
    per = 16 * L + 8
    sess = g.Session(model)
    toks = synth.tokens(V, PROMPT)
    d_prompt = torch.tensor(np.asarray(toks, np.int32), device="cuda")
    tout = torch.empty(LAST - PROMPT, dtype=torch.int32, device="cuda")
    assert sess.run(d_prompt, PROMPT, None, 0, tout) == "ok" and sess.sync() == "ok"
    tin = torch.full((LAST - PROMPT,), -1, dtype=torch.int32, device="cuda")
    tin[0] = int(tout[PROMPT - 1].item())
    logits = torch.empty(V, dtype=torch.float32, device="cuda")
    out = []
    for pos in sorted(positions):
        stamps = torch.zeros(8 + G * per, dtype=torch.int64, device="cuda")
        assert sess.rewind(pos) == "ok" and sess.set_timing(stamps) == "ok"
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        assert sess.run(tin, LAST - pos, logits, 0, tout) == "ok"
        e1.record()
        assert sess.sync() == "ok"
        torch.cuda.synchronize()
        a = stamps.cpu().numpy()
        R = a[8:].reshape(G, per)[:, :16 * L + 4].astype(np.float64)
        R[:, [16 * l + k for l in range(L) for k in range(10, 16)]] = 0
        t0 = R[R > 0].min()
        S = np.where(R > 0, R - t0, np.nan) / 1e3
        rel = np.array([[np.nanmax(S[:, 16 * l + k]) - np.nanmax(S[:, 16 * (l - 1) + 9]) for k in range(10)]
                        for l in range(1, L)]).mean(axis=0)
        spread = np.array([[np.nanmax(S[:, 16 * l + k]) - np.nanmin(S[:, 16 * l + k]) for k in range(10)]
                           for l in range(1, L)]).mean(axis=0)
        v = S[:, 16 * L:16 * L + 4]
        out.append({"position": pos, "status": sess.sync(), "us_per_step": 1e3 * e0.elapsed_time(e1) / (LAST - pos),
                    "gave_up": [int(x) for x in a[:6]],
                    "stage_end_us": dict(zip(STAGES, rel.round(2).tolist())),
                    "stage_spread_us": dict(zip(STAGES, spread.round(2).tolist())),
                    "layer_us": float(np.mean(np.diff([np.nanmax(S[:, 16 * l + 9]) for l in range(L)]))),
                    "vocab_us": float(np.nanmax(v[:, 3]) - np.nanmax(S[:, 16 * (L - 1) + 9]))})
    sess.close()
    model.close()
    return {"kernel": kind, "clusters": nc, "cluster_size": cs, "quant": quant, "runs": out}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--quant", choices=["f32", "f16"], default="f32")
    ap.add_argument("--positions", default="16,64,120")
    args = ap.parse_args()
    r = profile(args.quant, [int(x) for x in args.positions.split(",")])
    print(f"cluster step kernel: {r['clusters']} clusters of {r['cluster_size']} CTAs, {r['quant']}")
    for run in r["runs"]:
        print(f"run from position {run['position']}: {run['us_per_step']:.1f} us/step ({run['status']}); "
              f"layer {run['layer_us']:.2f} us, vocabulary stage {run['vocab_us']:.2f} us")
        print("  stage end after the previous layer (us): " +
              " ".join(f"{k}={v:.2f}" for k, v in run["stage_end_us"].items()))
        print("  spread over CTAs (us):                   " +
              " ".join(f"{k}={v:.2f}" for k, v in run["stage_spread_us"].items()))


if __name__ == "__main__":
    main()
