"""placeholder"""
def varlen_fwd(*a, **k): raise RuntimeError("not built")
def last_error(): return ""
def device_status(*a): raise RuntimeError("not built")
def library_path(): return None
class PaError(RuntimeError): pass
