"""Host-side logic of the torch.optim front end (no kernel runs): Philox
offsets are handed out in first-seen order, and a state_dict round trip keeps
every state tensor's dtype and the next free offset, and the AdamW front
ends pass their exact option on."""
import torch

from bit_blockwise_adamw_gb300 import optim


def _fake_state(opt, params):
    for p in params:
        st = opt.state[p]
        opt._offset(p, st)
        n = p.numel()
        st["m_codes"] = torch.arange(n, dtype=torch.int64).remainder(256).to(torch.uint8)
        st["m_absmax"] = torch.full(((n + 2047) // 2048,), 1.0 + 2 ** -20, dtype=torch.float32)
        st["m32"] = torch.full((n,), 1.0 + 2 ** -20, dtype=torch.float32)


def test_offsets_are_running_element_counts():
    ps = [torch.nn.Parameter(torch.zeros(n, dtype=torch.bfloat16)) for n in (5, 4096, 7)]
    opt = optim.Lion8bitSR(ps)
    assert [opt._offset(p, opt.state[p]) for p in ps] == [0, 5, 4101]
    assert opt._offset(ps[0], opt.state[ps[0]]) == 0     # stable once assigned


def test_state_dict_round_trip_keeps_dtypes():
    ps = [torch.nn.Parameter(torch.zeros(n, dtype=torch.bfloat16)) for n in (5000, 3)]
    opt = optim.AdamW8bitSR(ps)
    _fake_state(opt, ps)
    sd = opt.state_dict()
    qs = [torch.nn.Parameter(torch.zeros(n, dtype=torch.bfloat16)) for n in (5000, 3)]
    opt2 = optim.AdamW8bitSR(qs)
    opt2.load_state_dict(sd)
    for p, q in zip(ps, qs):
        for k in ("m_codes", "m_absmax", "m32"):
            a, b = opt.state[p][k], opt2.state[q][k]
            assert a.dtype == b.dtype and torch.equal(a, b)
    assert opt2._next_offset == 5003
    fresh = torch.nn.Parameter(torch.zeros(10, dtype=torch.bfloat16))
    opt2.add_param_group({"params": [fresh]})
    assert opt2._offset(fresh, opt2.state[fresh]) == 5003


def test_exact_option_reaches_the_hyper_parameters(monkeypatch):
    """AdamW front ends: exact=False (the default, fast mode) and exact=True
    reach q8_adamw_hparams.exact; a parameter group saved before the option
    existed (no "exact" key) runs in the fast mode."""
    seen = []
    monkeypatch.setattr(optim.B, "adamw8bit_sr_step", lambda arr, hp, *a: seen.append(hp.exact))
    monkeypatch.setattr(optim.B, "adamw_bf16_sr_step", lambda arr, hp, *a: seen.append(hp.exact))
    for cls in (optim.AdamW8bitSR, optim.AdamWBF16SR):
        for kw in ({}, {"exact": False}, {"exact": True}):
            opt = cls([torch.nn.Parameter(torch.zeros(8, dtype=torch.bfloat16))], **kw)
            group = opt.param_groups[0]
            group["step"] = 1
            opt._run(group, None)
        del group["exact"]
        opt._run(group, None)
    assert seen == [0, 0, 1, 0] * 2


def test_hparams_exact_field():
    import bit_blockwise_adamw_gb300 as q8
    assert q8.hparams().exact == 0 and q8.hparams(exact=1).exact == 1 and q8.hparams(exact=True).exact == 1
